"""Parity of the split chunked read (pa_decode_chunk_splitkv + pa_merge) with the oracle.

Every (sequence, query, head, split) partial output and lse is compared with
the fp64 oracle's chunk_splitkv_partials: the set of empty splits (lse -inf,
output 0) exactly, the rest within 2e-2 abs + 2e-2 rel; the merged rows
with paged_decode_chunk.  Cases run both kernels: mma.sync for small chunks,
tcgen05 from 64 (query, head) rows per kv head at head_dim 64 and from 128
rows at head_dim 128.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _q(base, n_q, seed=12, device="cpu"):
    g = torch.Generator(device=device).manual_seed(seed)
    b, hq, d = base.q.shape
    return torch.randn((b, n_q, hq, d), generator=g, device=device).to(base.dtype)


def _split(lib, g, q, pps, num_splits=None, err=None):
    s = num_splits or lib.pa_num_splits(g.max_blocks, pps)
    b, nq, hq, d = q.shape
    po = torch.full((b, nq, hq, s, d), float("nan"), device=DEV)
    pl = torch.full((b, nq, hq, s), float("nan"), device=DEV)
    lib.pa_decode_chunk_splitkv(po, pl, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                g.scale, pps, dev_err=err)
    out = torch.empty_like(q)
    lib.pa_merge(out, po, pl)
    torch.cuda.synchronize()
    return po, pl, out


def _oracle_partials(base, q, pps, s, seqs=None):
    idx = list(range(base.num_seqs) if seqs is None else seqs)
    return oracle.chunk_splitkv_partials(host_f32(q[idx]), host_f32(base.k_pool),
                                         host_f32(base.v_pool), base.block_table[idx].numpy(),
                                         base.seq_lens[idx].numpy(), base.scale,
                                         base.block_size, pps, s)


def _oracle_chunk(base, q, seqs=None):
    idx = list(range(base.num_seqs) if seqs is None else seqs)
    return oracle.paged_decode_chunk(host_f32(q[idx]), host_f32(base.k_pool),
                                     host_f32(base.v_pool), base.block_table[idx].numpy(),
                                     base.seq_lens[idx].numpy(), base.scale, base.block_size)


def _check_partials(po, pl, ref_po, ref_pl, dtype, what=""):
    got_l = pl.double().cpu().numpy()
    assert np.array_equal(np.isneginf(got_l), np.isneginf(ref_pl)), f"{what}: empty splits differ"
    empty = np.isneginf(ref_pl)
    assert torch.all(po.cpu()[torch.from_numpy(empty)] == 0), f"{what}: empty split not zero"
    fin = ~empty
    err = np.abs(got_l[fin] - ref_pl[fin])
    assert np.all(err <= 2e-2 + 2e-2 * np.abs(ref_pl[fin])), f"{what}: lse max err {err.max()}"
    assert_attn_close(po, ref_po, dtype, f"{what} partials")


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,n_q,lens,pps", [
    ("bf16", 32, 8, 64, 16, 4, [4, 37, 300, 1000], 2),       # 16 rows: mma.sync
    ("f16", 12, 4, 48, 16, 7, [7, 13, 100, 257], 1),         # group 3, head_dim 48
    ("bf16", 32, 8, 128, 16, 8, [8, 65, 700, 1500], 5),      # 32 rows, head_dim 128
    ("bf16", 32, 8, 64, 16, 16, [16, 40, 333, 1200], 3),     # 64 rows: tcgen05
    ("bf16", 32, 8, 64, 16, 50, [50, 70, 640, 900], 4),      # 200 rows: two tiles
    ("f16", 32, 8, 128, 8, 32, [32, 33, 129, 1000], 16),     # fp16, pages of 8
    ("bf16", 32, 2, 128, 16, 8, [8, 9, 250, 3000], 7),       # group 16: 128 rows
    ("bf16", 16, 4, 64, 16, 48, [20, 48, 130, 640], 1),      # queries at negative positions
    ("bf16", 32, 8, 64, 16, 80, [80, 90, 700, 1300], 3),     # 320 rows: warp-specialized
    ("f16", 32, 8, 128, 16, 64, [64, 200, 900, 1100], 8),    # 256 rows, head_dim 128
    ("bf16", 32, 8, 64, 128, 64, [64, 300, 1000, 1500], 1),  # pages of 128, one per split
    ("bf16", 32, 8, 64, 16, 64, [64, 300, 1000, 1500], 5),   # splits of 80 tokens: tiles off 64
    ("f16", 32, 8, 128, 16, 2, [3, 50, 700, 1600], 2),       # 8 columns on the decode kernel
    ("bf16", 32, 4, 64, 16, 2, [1, 40, 333, 1200], 3),       # group 8, a query at position -1
    ("bf16", 8, 8, 64, 16, 16, [16, 300, 900, 1111], 4),     # group 1: 16 queries, one head each
    ("bf16", 12, 3, 64, 16, 16, [16, 40, 3000, 1200, 5], 2),  # 64 rows, 15 (seq, kv head) pairs
    ("f16", 8, 1, 64, 16, 12, [12, 900, 1300], 9),           # 96 rows, one kv head
    ("bf16", 32, 8, 64, 16, 100, [100, 110, 400], 4),        # 400 rows, a long chunk: one Q tile
                                                             # per CTA at head_dim 64
])
def test_partials_and_merge(lib, dtype, hq, hkv, d, bs, n_q, lens, pps):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("chunk_split", 51, dtype, lens, hq, hkv, d, bs, pages)
    q = _q(base, n_q)
    g = base.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    po, pl, out = _split(lib, g, q.to(DEV), pps, err=err)
    assert int(err.item()) == 0
    ref_po, ref_pl = _oracle_partials(base, q, pps, po.shape[3])
    _check_partials(po, pl, ref_po, ref_pl, base.dtype, f"pps {pps}")
    assert_attn_close(out, _oracle_chunk(base, q), base.dtype, "merged")


def test_split_merge_matches_the_one_pass_read(lib):
    base = workloads.make_batch("chunk_split_eq", 52, "bf16", [100, 900, 2000, 64], 32, 8, 64,
                                16, 260)
    g = base.to(DEV)
    for n_q in (3, 16, 40):
        q = _q(base, n_q, seed=n_q).to(DEV)
        one = torch.empty_like(q)
        lib.pa_decode_chunk(one, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale)
        _, _, out = _split(lib, g, q, 8)
        assert torch.allclose(out.float(), one.float(), atol=2e-2, rtol=2e-2), n_q


def test_extra_splits_are_empty(lib):
    base = workloads.make_batch("chunk_split_extra", 53, "bf16", [30, 200], 32, 8, 64, 16, 20)
    q = _q(base, 16)
    g = base.to(DEV)
    need = lib.pa_num_splits(g.max_blocks, 4)
    po, pl, out = _split(lib, g, q.to(DEV), 4, num_splits=need + 3)
    assert torch.isneginf(pl[..., need:]).all() and torch.all(po[..., need:, :] == 0)
    assert_attn_close(out, _oracle_chunk(base, q), base.dtype)


@pytest.mark.parametrize("n_q", [4, 16])
def test_bad_page_zeroes_only_its_split(lib, n_q):
    base = workloads.make_batch("chunk_split_bad", 54, "bf16", [600, 800], 32, 8, 64, 16, 100)
    q = _q(base, n_q)
    good = base.block_table.clone()
    base.block_table[1, 9] = base.num_pages + 4      # page 9: split 4 at 2 pages per split
    g = base.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    po, pl, _ = _split(lib, g, q.to(DEV), 2, err=err)
    assert int(err.item()) == 1
    assert torch.isneginf(pl[1, :, :, 4]).all() and torch.all(po[1, :, :, 4] == 0)
    base.block_table = good
    ref_po, ref_pl = _oracle_partials(base, q, 2, po.shape[3])
    keep = [s for s in range(po.shape[3]) if s != 4]
    _check_partials(po[0], pl[0], ref_po[0], ref_pl[0], base.dtype, "seq 0")
    _check_partials(po[1][:, :, keep], pl[1][:, :, keep], ref_po[1][:, :, keep],
                    ref_pl[1][:, :, keep], base.dtype, "seq 1")


@pytest.mark.parametrize("n_q", [4, 16])
def test_longctx_32k_sampled(lib, n_q):
    # the long-context chunk: 2 sequences x 32,768 tokens, head_dim 128, 1% of keys x8,
    # 64 pages per split; sampled queries against attention over their causal prefixes
    g = workloads.longctx(32768, batch=2, device=DEV)
    q = _q(g, n_q, seed=5, device=DEV)
    _, _, out = _split(lib, g, q, 64)
    n = 32768
    for b in (0, 1):
        pages = g.block_table[b].long()
        k = host_f32(g.k_pool.index_select(0, pages)).reshape(n, 8, 128)
        v = host_f32(g.v_pool.index_select(0, pages)).reshape(n, 8, 128)
        for i in (0, n_q - 1):
            seen = n - n_q + i + 1
            for h in (0, 13, 31):
                ref, _ = oracle.attend(host_f32(q[b, i, h]), k[:seen, h // 4], v[:seen, h // 4],
                                       g.scale)
                assert_attn_close(out[b, i, h], ref, g.dtype, f"b{b} i{i} h{h}")


def test_small_chunk_many_splits_per_cta(lib):
    # few (sequence, kv head) pairs and many splits: the decode kernel covers several
    # consecutive splits per CTA, here with 2 queries x 4 heads per kv head
    base = workloads.make_batch("chunk_multi", 55, "bf16", [8192, 5000], 16, 4, 128, 16, 900)
    q = _q(base, 2)
    g = base.to(DEV)
    po, pl, out = _split(lib, g, q.to(DEV), 2)
    ref_po, ref_pl = _oracle_partials(base, q, 2, po.shape[3])
    _check_partials(po, pl, ref_po, ref_pl, base.dtype, "many splits")
    assert_attn_close(out, _oracle_chunk(base, q), base.dtype, "merged")
