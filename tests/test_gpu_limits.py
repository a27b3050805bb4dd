"""Parity at the limits the C ABI's host checks accept.

The host layer takes block_size up to 1024, num_seqs up to 65,535 (the grid's
y extent) and any split count whose grid fits.  Each case here is an ordinary
call at such a limit, compared element by element with the fp64 oracle:

* block_size 1024 on every read path: the single-pass read (tensor-core and
  CUDA-core), the split read + merge, and the chunked read on each of its
  kernels (the decode kernel's chunk mode, the pipelined one-tile and the
  warp-specialized tcgen05 reads) and its split form;
* 65,535 sequences of short histories, single pass and split + merge;
* merges over 20,000+ splits: one sequence of 327,680 tokens split into
  one-page runs (through the split read), and random partials with empty
  splits (pa_merge alone).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"

# histories around the 1024-token page: one token, a page less one, one page, one page and
# one token, and several pages with a ragged tail
BS1024_LENS = [1, 1023, 1024, 1025, 2500, 4097]


def _pages_f64(batch, b):
    """Float64 host copies of sequence b's pages and a renumbered table row."""
    n = int(batch.seq_lens[b])
    npg = -(-n // batch.block_size)
    pages = batch.block_table[b, :npg].long().to(batch.k_pool.device)
    k = batch.k_pool.index_select(0, pages).double().cpu().numpy()
    v = batch.v_pool.index_select(0, pages).double().cpu().numpy()
    return k, v, np.arange(npg), n


def _ref_decode(batch, seqs=None):
    seqs = range(batch.num_seqs) if seqs is None else seqs
    out = []
    for b in seqs:
        k, v, row, n = _pages_f64(batch, b)
        out.append(oracle.paged_decode_one(batch.q[b].double().cpu().numpy(), k, v, row, n,
                                           batch.scale, batch.block_size))
    return np.stack(out)


def _split(lib, g, pps):
    s = lib.pa_num_splits(g.max_blocks, pps)
    b, hq, d = g.q.shape
    po = torch.full((b, hq, s, d), float("nan"), device=DEV)
    pl = torch.full((b, hq, s), float("nan"), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                          pps, dev_err=err)
    out = torch.empty_like(g.q)
    lib.pa_merge(out, po, pl)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return po, pl, out


# ---------------------------------------------------------------- block_size 1024


@pytest.mark.parametrize("dtype,hq,hkv,d", [("bf16", 8, 2, 64), ("f16", 12, 4, 48),
                                             ("bf16", 16, 2, 128), ("f32", 8, 2, 64)])
def test_block_size_1024_single_pass_and_split(lib, dtype, hq, hkv, d):
    pages = sum(-(-n // 1024) for n in BS1024_LENS) + 3
    g = workloads.make_batch("bs1024", 71, dtype, BS1024_LENS, hq, hkv, d, 1024,
                             pages).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty_like(g.q)
    lib.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = _ref_decode(g)
    assert_attn_close(out, ref, g.dtype, "single pass")
    for pps in (1, 2):
        po, pl, merged = _split(lib, g, pps)
        assert_attn_close(merged, ref, g.dtype, f"split {pps} + merge")
        for b in (1, 5):                          # partials of two sequences
            k, v, row, n = _pages_f64(g, b)
            rpo, rpl = oracle.splitkv_partials(g.q[b:b + 1].double().cpu().numpy(), k, v,
                                               row[None, :], np.array([n]), g.scale, 1024, pps,
                                               po.shape[2])
            assert_attn_close(po[b], rpo[0], g.dtype, f"partials seq {b} pps {pps}")
            got = pl[b].cpu().double().numpy()
            tol = 1e-5 if dtype == "f32" else 2e-2
            finite = np.isfinite(rpl[0])
            assert np.array_equal(np.isfinite(got), finite)
            assert np.all(np.abs(got[finite] - rpl[0][finite]) <= tol + tol * np.abs(rpl[0][finite]))


@pytest.mark.parametrize("d,n_q", [(64, 4), (64, 8), (64, 32), (64, 64), (128, 2), (128, 64)])
def test_block_size_1024_chunked_read_and_its_splits(lib, d, n_q):
    # G = 4: n_q * 4 rows per kv head reach the decode kernel's chunk mode (<= 16 at head_dim
    # 64, <= 8 at 128), the pipelined one-tile tcgen05 read (32, 128) and the warp-specialized
    # one (256)
    lens = [max(n_q, x) for x in (70, 1023, 1024, 1025, 2500)]
    pages = sum(-(-n // 1024) for n in lens) + 2
    g = workloads.make_batch("bs1024c", 72, "bf16", lens, 16, 4, d, 1024, pages).to(DEV)
    gen = torch.Generator().manual_seed(5)
    q = torch.randn((g.num_seqs, n_q, 16, d), generator=gen).to(torch.bfloat16).to(DEV)
    out = torch.full_like(q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_decode_chunk(out, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                        dev_err=err)
    s = lib.pa_num_splits(g.max_blocks, 1)
    po = torch.full((g.num_seqs, n_q, 16, s, d), float("nan"), device=DEV)
    pl = torch.full((g.num_seqs, n_q, 16, s), float("nan"), device=DEV)
    lib.pa_decode_chunk_splitkv(po, pl, q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                                1, dev_err=err)
    merged = torch.empty_like(q)
    lib.pa_merge(merged, po, pl)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(g.num_seqs):
        k, v, row, n = _pages_f64(g, b)
        ref = oracle.paged_decode_chunk(q[b:b + 1].double().cpu().numpy(), k, v, row[None, :],
                                        np.array([n]), g.scale, 1024)
        assert_attn_close(out[b:b + 1], ref, g.dtype, f"chunk seq {b}")
        assert_attn_close(merged[b:b + 1], ref, g.dtype, f"chunk split + merge seq {b}")


# ---------------------------------------------------------------- 65,535 sequences


def test_the_largest_batch(lib):
    # every grid row: 65,535 sequences of 1-40 tokens, GQA 4, head_dim 64, bf16
    gen = torch.Generator().manual_seed(17)
    lens = torch.randint(1, 41, (65535,), generator=gen).tolist()
    pages = sum(-(-n // 16) for n in lens) + 16
    cpu = workloads.make_batch("b65535", 73, "bf16", lens, 4, 1, 64, 16, pages)
    g = cpu.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_cache_append(g.k_new, g.v_new, g.k_pool, g.v_pool, g.block_table, g.positions,
                        dev_err=err)
    out = torch.empty_like(g.q)
    lib.pa_decode(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _, _, merged = _split(lib, g, 1)
    # the oracle over the whole batch, on host copies with the append applied
    k2, v2 = oracle.cache_append(host_f32(cpu.k_pool), host_f32(cpu.v_pool), host_f32(cpu.k_new),
                                 host_f32(cpu.v_new), cpu.block_table.numpy(),
                                 cpu.positions.numpy(), 16)
    assert np.array_equal(host_f32(g.k_pool), k2)       # the append, bit for bit
    ref = oracle.paged_decode(host_f32(cpu.q), k2, v2, cpu.block_table.numpy(),
                              cpu.seq_lens.numpy(), cpu.scale, 16)
    assert_attn_close(out, ref, cpu.dtype, "single pass, 65,535 sequences")
    assert_attn_close(merged, ref, cpu.dtype, "split + merge, 65,535 sequences")


# ---------------------------------------------------------------- tens of thousands of splits


def test_twenty_thousand_one_page_splits(lib):
    # one sequence of 20,480 pages (327,680 tokens), one page per split: the split read
    # writes 20,480 partials per head and pa_merge combines them
    n = 20480 * 16
    g = workloads.make_batch("s20k", 74, "bf16", [n], 4, 1, 64, 16, 20480 + 8).to(DEV)
    po, pl, merged = _split(lib, g, 1)
    assert po.shape[2] == 20480
    assert_attn_close(merged, _ref_decode(g), g.dtype, "20,480 splits merged")
    # partials of a few splits, each a one-page attention
    k, v, row, _ = _pages_f64(g, 0)
    q0 = g.q[0].double().cpu().numpy()
    for s_ in (0, 1, 9999, 20479):
        for h in range(4):
            ro, rl = oracle.attend(q0[h], k[s_, :, 0, :], v[s_, :, 0, :], g.scale)
            assert_attn_close(po[0, h, s_], ro, g.dtype, f"split {s_} head {h}")
            assert abs(float(pl[0, h, s_]) - rl) <= 2e-2 + 2e-2 * abs(rl)


@pytest.mark.parametrize("splits", [20000, 65535])
def test_merge_of_many_random_partials(lib, splits):
    # pa_merge alone on random partials: lse spread over [-30, 30] with a quarter of the
    # splits empty (-inf), one row with every split empty
    gen = torch.Generator().manual_seed(splits)
    b, hq, d = 2, 4, 64
    po = torch.randn((b, hq, splits, d), generator=gen)
    pl = torch.rand((b, hq, splits), generator=gen) * 60 - 30
    pl[torch.rand((b, hq, splits), generator=gen) < 0.25] = -float("inf")
    pl[1, 3] = -float("inf")
    out = torch.empty((b, hq, d), dtype=torch.bfloat16, device=DEV)
    lib.pa_merge(out, po.to(DEV), pl.to(DEV))
    ref = oracle.merge_partials(po.double().numpy(), pl.double().numpy())
    torch.cuda.synchronize()
    assert_attn_close(out, ref, torch.bfloat16, f"merge over {splits} splits")
    assert torch.all(out[1, 3] == 0)
