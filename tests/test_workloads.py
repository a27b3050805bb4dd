"""The seeded input recipe: determinism, block-table structure and the named
shapes, checked on the CPU at reduced sizes (the same code draws the full
sizes, on the device for the two largest)."""

import math

import pytest
import torch

import workloads


def _tables_are_disjoint_runs(batch):
    """Each sequence owns ceil(len / bs) distinct in-range pages, no page is shared, and the
    entries past them are -1."""
    seen = set()
    for b, n in enumerate(batch.lens_list()):
        need = math.ceil(n / batch.block_size)
        row = batch.block_table[b].tolist()
        pages = row[:need]
        assert all(0 <= p < batch.num_pages for p in pages)
        assert all(p == -1 for p in row[need:])
        assert not seen.intersection(pages) and len(set(pages)) == need
        seen.update(pages)


def test_same_seed_same_batch_and_tables_are_not_contiguous():
    a, b = workloads.awkward(), workloads.awkward()
    for name in ("q", "k_pool", "v_pool", "block_table", "seq_lens", "k_new", "v_new"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    _tables_are_disjoint_runs(a)
    row = a.block_table[3, :17].tolist()
    assert row != sorted(row)                     # a permutation, not pages in order


def test_a_different_seed_draws_different_numbers():
    a = workloads.make_batch("x", 10, "bf16", [40, 70], 8, 2, 64, 16, 20)
    b = workloads.make_batch("x", 11, "bf16", [40, 70], 8, 2, 64, 16, 20)
    assert not torch.equal(a.k_pool, b.k_pool) and not torch.equal(a.q, b.q)


def test_named_shapes():
    t = workloads.tiny()
    assert (t.num_seqs, t.num_q_heads, t.num_kv_heads, t.head_dim, t.block_size) == (1, 32, 8, 64, 16)
    assert t.dtype == torch.float32 and t.num_pages == 16 and t.lens_list() == [64]
    w = workloads.awkward()
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.dtype) == (12, 4, 48, torch.float16)
    assert w.lens_list() == [1, 13, 100, 257]
    lm = workloads.llama1b(1024, batch=4, num_pages=300)
    assert (lm.num_seqs, lm.num_q_heads, lm.num_kv_heads, lm.head_dim) == (4, 32, 8, 64)
    assert lm.dtype == torch.bfloat16 and lm.lens_list() == [1024] * 4
    assert lm.scale == pytest.approx(1 / 8)
    _tables_are_disjoint_runs(lm)
    # the appended token sits at the last attended position
    assert torch.equal(lm.positions, lm.seq_lens - 1)
    assert lm.k_new.shape == (4, 8, 64) and lm.v_new.shape == (4, 8, 64)


def test_ragged_lengths_are_uniform_in_range_with_std_half():
    r = workloads.ragged8b(batch=32, num_pages=1200, max_len=512)
    lens = r.lens_list()
    assert all(16 <= n <= 512 for n in lens) and len(set(lens)) > 16
    assert (r.num_q_heads, r.num_kv_heads, r.head_dim) == (32, 8, 128)
    _tables_are_disjoint_runs(r)
    assert r.k_pool.float().std().item() == pytest.approx(0.5, rel=0.02)


def test_longctx_scales_about_one_percent_of_keys_by_eight():
    g = workloads.longctx(4096, batch=2)
    assert g.num_pages == 2 * 4096 // 16          # exactly the pages needed
    tokens = 2 * 4096
    n = g.meta["n_peaky"]
    assert abs(n - 0.01 * tokens) < 5 * math.sqrt(0.01 * tokens)
    # a scaled key row has a standard deviation near 8, the others near 1
    k = g.k_pool.float().reshape(-1, g.num_kv_heads * g.head_dim)
    big = (k.std(dim=1) > 4).sum().item()
    assert big == n


def test_dense_cache_is_the_identity_table():
    d = workloads.dense(1024, batch=2)
    assert torch.equal(d.block_table.flatten(), torch.arange(2 * 64, dtype=torch.int32))
    assert d.lens_list() == [1024, 1024] and d.dtype == torch.float16
    assert (d.num_q_heads, d.num_kv_heads, d.head_dim) == (16, 16, 64)
