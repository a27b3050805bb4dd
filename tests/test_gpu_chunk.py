"""Parity of the chunked multi-query read (pa_decode_chunk) with the oracle.

Each sequence's chunk of queries was appended before the read; query i
sits at position seq_len - chunk_len + i and attends causally.  Compared
with the fp64 oracle's paged_decode_chunk, elementwise within 2e-2 abs +
2e-2 rel (f16/bf16).
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_attn_close, host_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _chunk_batch(base, n_q, seed=11):
    """The base batch with a chunk of n_q queries per sequence instead of one."""
    g = torch.Generator().manual_seed(seed)
    b, hq, d = base.q.shape
    q = torch.randn((b, n_q, hq, d), generator=g).to(base.dtype)
    return q


def _run(lib, base, q, dev_err=None):
    gpu = base.to(DEV)
    qd = q.to(DEV)
    out = torch.full_like(qd, float("nan"))
    lib.pa_decode_chunk(out, qd, gpu.k_pool, gpu.v_pool, gpu.block_table, gpu.seq_lens, base.scale,
                        dev_err=dev_err)
    return out


def _ref(base, q, seqs=None):
    seqs = range(base.num_seqs) if seqs is None else seqs
    idx = list(seqs)
    return oracle.paged_decode_chunk(host_f32(q[idx]), host_f32(base.k_pool), host_f32(base.v_pool),
                                     base.block_table[idx].numpy(), base.seq_lens[idx].numpy(),
                                     base.scale, base.block_size)


@pytest.mark.parametrize("n_q", [1, 3, 8, 16, 40])
def test_awkward_chunks(lib, n_q):
    # histories {1, 13, 100, 257}, group 3, head_dim 48, fp16; chunks longer than
    # a history put queries at negative positions (output 0)
    base = workloads.awkward()
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype, f"n_q={n_q}")


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,n_q", [
    ("bf16", 32, 8, 64, 16, 16),
    ("bf16", 32, 8, 128, 16, 7),
    ("f16", 16, 2, 64, 1, 9),        # group 8, one token per page
    ("bf16", 32, 2, 32, 64, 5),      # group 16, big pages
    ("bf16", 8, 8, 96, 8, 33),       # group 1: 33 rows per kv head
])
def test_shapes(lib, dtype, hq, hkv, d, bs, n_q):
    lens = [n_q, n_q + 1, 3 * bs + 7, 300]
    pages = sum(-(-n // bs) for n in lens) + 3
    base = workloads.make_batch("chunk", 23, dtype, lens, hq, hkv, d, bs, pages)
    q = _chunk_batch(base, n_q)
    out = _run(lib, base, q)
    assert_attn_close(out, _ref(base, q), base.dtype)


def test_one_query_chunk_matches_the_single_query_read(lib):
    base = workloads.llama1b(256, batch=8)
    gpu = base.to(DEV)
    out = _run(lib, base, base.q.unsqueeze(1))[:, 0]
    single = torch.empty_like(gpu.q)
    lib.pa_decode(single, gpu.q, gpu.k_pool, gpu.v_pool, gpu.block_table, gpu.seq_lens, base.scale)
    assert_attn_close(out, single.double().cpu().numpy(), base.dtype)


def test_llama1b_h4096_chunk16_sampled(lib):
    # the measured launch: 64 sequences, 16-query chunks at history 4096
    base = workloads.llama1b(4096)
    q = _chunk_batch(base, 16)
    out = _run(lib, base, q)
    torch.cuda.synchronize()
    for b in (0, 63):
        assert_attn_close(out[b:b + 1], _ref(base, q, [b]), base.dtype, f"seq {b}")


def test_bad_page_is_reported_and_zeroed(lib):
    base = workloads.awkward()
    base.block_table[3, 1] = -7
    q = _chunk_batch(base, 4)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[3] == 0)
    assert_attn_close(out[:3], _ref(base, q, [0, 1, 2]), base.dtype)


@pytest.mark.parametrize("scale", [-0.125, 0.0, 0.7])
def test_any_finite_scale(lib, scale):
    # a negative scale runs as a sign flip of q; scale 0 gives the mean of the visible V rows
    base = workloads.awkward()
    base.scale = scale
    q = _chunk_batch(base, 5)
    out = _run(lib, base, q)
    assert_attn_close(out, _ref(base, q), base.dtype, f"scale {scale}")


# ------------------------------------------- tcgen05 path (>= 64 rows at d 64, 128 at d 128)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,n_q,lens", [
    ("bf16", 32, 8, 64, 16, 32, [32, 100, 700, 4096]),       # 128 rows: one tile
    ("bf16", 32, 8, 64, 16, 50, [60, 50, 333, 1000]),        # 200 rows: a partial second tile
    ("bf16", 32, 8, 128, 16, 40, [40, 41, 500, 2049]),       # head_dim 128
    ("f16", 32, 8, 128, 8, 64, [64, 65, 129, 900]),          # fp16, pages of 8
    ("bf16", 32, 4, 64, 32, 16, [16, 300, 777, 1500]),       # group 8
    ("bf16", 32, 2, 128, 16, 8, [8, 9, 250, 3000]),          # group 16
    ("f16", 16, 4, 64, 16, 48, [20, 48, 130, 640]),          # queries at negative positions
])
def test_tensor_core_chunks(lib, dtype, hq, hkv, d, bs, n_q, lens):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("tc", 41, dtype, lens, hq, hkv, d, bs, pages)
    assert n_q * (hq // hkv) >= 128
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


# 64-128 (query, head) rows per kv head at head_dim 64 (the pipelined one-tile tcgen05 read):
# an empty sequence, lengths far apart, odd (sequence, kv head) counts, odd page sizes
@pytest.mark.parametrize("dtype,hq,hkv,bs,n_q,lens", [
    ("bf16", 12, 3, 16, 16, [0, 16, 4000, 1500, 77]),      # 15 (sequence, kv head) pairs
    ("f16", 8, 8, 16, 100, [100, 101, 2500]),              # group 1, 100 rows
    ("bf16", 32, 4, 8, 16, [16, 3000, 200]),               # group 8, 128 rows, pages of 8
    ("bf16", 4, 1, 1024, 20, [20, 2100, 1024, 1025]),      # one kv head, pages of 1024
    ("bf16", 8, 2, 4, 32, [32, 700, 33]),                  # pages of 4
])
def test_chunks_of_64_to_128_rows(lib, dtype, hq, hkv, bs, n_q, lens):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("pair", 46, dtype, lens, hq, hkv, 64, bs, pages)
    assert 64 <= n_q * (hq // hkv) <= 128
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


# 9-255 rows per kv head at head_dim 128 (the pipelined one-tile read): pages smaller than,
# equal to and larger than its 32-token key tile, an empty and a one-token sequence, odd
# and single kv-head counts
@pytest.mark.parametrize("dtype,hq,hkv,bs,n_q,lens", [
    ("bf16", 32, 8, 16, 16, [0, 16, 900, 2049]),            # 64 rows, pages of 16
    ("f16", 32, 8, 64, 24, [24, 25, 700, 1500]),            # 96 rows, pages of 64
    ("bf16", 16, 4, 1024, 30, [30, 1, 1100, 2050]),         # 120 rows, pages of 1024
    ("bf16", 32, 8, 4, 5, [5, 40, 333, 777]),               # 20 rows, pages of 4 (cp.async)
    ("f16", 32, 8, 32, 40, [40, 64, 500, 1600]),            # 160 rows, pages of 32: two Q tiles
    ("bf16", 12, 3, 16, 8, [8, 0, 300, 1025, 77]),          # 32 rows, three kv heads
    ("f16", 8, 8, 8, 48, [48, 49, 600]),                    # 48 rows (group 1)
    ("bf16", 4, 1, 16, 12, [12, 500, 13]),                  # 48 rows, one kv head
])
def test_pipelined_chunks_at_head_dim_128(lib, dtype, hq, hkv, bs, n_q, lens):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("pipe128", 48, dtype, lens, hq, hkv, 128, bs, pages)
    assert 9 <= n_q * (hq // hkv) < 256
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


def test_chunk_of_64_rows_bad_page_zeroes_only_its_sequence(lib):
    # one kv head, 16 queries x 4 heads; only sequence 0's table is bad
    base = workloads.make_batch("pairbad", 47, "bf16", [500, 700, 300], 4, 1, 64, 16, 120)
    base.block_table[0, 5] = -7
    q = _chunk_batch(base, 16)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[0] == 0)
    assert_attn_close(out[1:], _ref(base, q, [1, 2]), base.dtype)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f16", 64), ("bf16", 64)])
def test_tensor_core_prefill(lib, dtype, d):
    # whole prompts: chunk_len == seq_len, so past == 0 and the read is causal prefill
    # (head_dim 128: two Q tiles per CTA; head_dim 64: the pipelined one-tile read)
    base = workloads.make_batch("prefill", 43, dtype, [200, 200, 200], 32, 8, d, 16, 40)
    q = _chunk_batch(base, 200)
    out = _run(lib, base, q)
    assert_attn_close(out, _ref(base, q), base.dtype, "prefill")


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.6])
def test_tensor_core_any_finite_scale(lib, scale):
    base = workloads.make_batch("tcs", 44, "bf16", [64, 300, 90], 32, 8, 64, 16, 40)
    base.scale = scale
    q = _chunk_batch(base, 32)
    out = _run(lib, base, q)
    assert_attn_close(out, _ref(base, q), base.dtype, f"scale {scale}")


def test_tensor_core_bad_page_is_reported_and_zeroed(lib):
    base = workloads.make_batch("tcbad", 45, "bf16", [64, 300, 500], 32, 8, 64, 16, 60)
    base.block_table[2, 3] = base.num_pages + 9
    q = _chunk_batch(base, 32)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[2] == 0)
    assert_attn_close(out[:2], _ref(base, q, [0, 1]), base.dtype)


@pytest.mark.parametrize("d", [64, 128])   # the pipelined one-tile read; two Q tiles per CTA
def test_prefill_4096_whole_prompt_and_sampled_rows(lib, d):
    # the measured prefill launch (8 prompts x 4096 tokens): one whole prompt (every query
    # and head) against the oracle's chunked read, and sampled queries of two more prompts
    # against attention over their causal prefixes
    base = workloads.make_batch(f"prefill_d{d}", 6, "bf16", [4096] * 8, 32, 8, d, 16, 8 * 256,
                                device=DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(8)
    q = torch.randn((8, 4096, 32, d), generator=gen, device=DEV).to(torch.bfloat16)
    out = torch.empty_like(q)
    lib.pa_decode_chunk(out, q, base.k_pool, base.v_pool, base.block_table, base.seq_lens,
                        base.scale)
    torch.cuda.synchronize()
    for b in (0, 7):
        pages = base.block_table[b].long()
        k = host_f32(base.k_pool.index_select(0, pages)).reshape(4096, 8, d)
        v = host_f32(base.v_pool.index_select(0, pages)).reshape(4096, 8, d)
        for i in (0, 1, 127, 128, 2000, 4095):
            for h in (0, 5, 31):
                ref, _ = oracle.attend(host_f32(q[b, i, h]), k[:i + 1, h // 4], v[:i + 1, h // 4],
                                       base.scale)
                assert_attn_close(out[b, i, h], ref, base.dtype, f"b{b} i{i} h{h}")
    # prompt 3 whole: the oracle's chunked read, one kv head (and its 4 query heads) at a
    # time on float64 copies of the prompt's pages (heads are independent in the definition)
    b = 3
    pages = base.block_table[b].long()
    kp = base.k_pool.index_select(0, pages).double().cpu().numpy()     # [256, 16, 8, d]
    vp = base.v_pool.index_select(0, pages).double().cpu().numpy()
    qb = q[b:b + 1].double().cpu().numpy()                              # [1, 4096, 32, d]
    got = out[b:b + 1]
    for g in range(8):
        ref = oracle.paged_decode_chunk(np.ascontiguousarray(qb[:, :, 4 * g:4 * g + 4]),
                                        np.ascontiguousarray(kp[:, :, g:g + 1]),
                                        np.ascontiguousarray(vp[:, :, g:g + 1]),
                                        np.arange(256)[None, :], np.array([4096]), base.scale, 16)
        assert_attn_close(got[:, :, 4 * g:4 * g + 4], ref, base.dtype, f"prompt 3 kv head {g}")


# ------------------------------- warp-specialized tcgen05 path (>= 256 rows per kv head)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,n_q,lens", [
    ("bf16", 32, 8, 64, 16, 64, [64, 100, 700, 1000]),       # 256 rows: one CTA, two Q tiles
    ("bf16", 32, 8, 64, 16, 100, [100, 130, 640, 2000]),     # 400 rows: second CTA's tile 1 partial
    ("bf16", 32, 8, 128, 16, 80, [80, 81, 333, 1500]),       # 320 rows: second CTA's tile 1 empty
    ("f16", 32, 8, 64, 8, 72, [72, 73, 200, 900]),           # fp16, pages of 8
    ("bf16", 32, 2, 128, 16, 16, [16, 17, 300, 2500]),       # group 16
    ("f16", 16, 4, 64, 16, 96, [30, 96, 200, 700]),          # queries at negative positions
    ("bf16", 32, 8, 64, 32, 128, [128, 129, 1024, 4096]),    # 512 rows, pages of 32
    ("bf16", 32, 8, 64, 128, 64, [64, 300, 1000, 1500]),     # pages of 128: two copies per page
    ("f16", 32, 8, 128, 256, 80, [80, 500, 700, 1300]),      # pages of 256, head_dim 128
    ("bf16", 32, 8, 64, 4, 64, [64, 99, 300, 650]),          # pages of 4: cp.async for every tile
])
def test_warp_specialized_chunks(lib, dtype, hq, hkv, d, bs, n_q, lens):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("ws", 46, dtype, lens, hq, hkv, d, bs, pages)
    assert n_q * (hq // hkv) >= 256
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


@pytest.mark.parametrize("scale", [-0.09, 0.0, 0.6])
def test_warp_specialized_any_finite_scale(lib, scale):
    base = workloads.make_batch("wss", 47, "bf16", [64, 300, 90], 32, 8, 64, 16, 40)
    base.scale = scale
    q = _chunk_batch(base, 64)
    out = _run(lib, base, q)
    assert_attn_close(out, _ref(base, q), base.dtype, f"scale {scale}")


def test_warp_specialized_bad_page_is_reported_and_zeroed(lib):
    base = workloads.make_batch("wsbad", 48, "bf16", [256, 300, 500], 32, 8, 128, 16, 80)
    base.block_table[2, 5] = -3
    q = _chunk_batch(base, 64)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[2] == 0)
    assert_attn_close(out[:2], _ref(base, q, [0, 1]), base.dtype)


# ---- up to 16 (query, head) columns per kv head (8 at head_dim 128): the decode kernel, per-column limits


@pytest.mark.parametrize("dtype,hq,hkv,d,bs,n_q,lens", [
    ("bf16", 32, 8, 64, 16, 2, [2, 37, 300, 1000]),          # 8 columns
    ("bf16", 32, 8, 64, 16, 3, [3, 16, 17, 2049]),           # 12 columns
    ("f16", 32, 8, 128, 16, 2, [2, 5, 640, 1500]),           # 8 columns, head_dim 128
    ("bf16", 32, 4, 64, 8, 2, [9, 64, 65, 700]),             # group 8: 16 columns, pages of 8
    ("bf16", 16, 8, 128, 32, 4, [1, 2, 100, 900]),           # group 2; queries at negative positions
    ("bf16", 8, 8, 64, 16, 16, [16, 17, 500, 1234]),         # group 1: 16 queries, one head each
])
def test_small_chunks_on_the_decode_kernel(lib, dtype, hq, hkv, d, bs, n_q, lens):
    pages = sum(-(-n // bs) for n in lens) + 5
    base = workloads.make_batch("small", 49, dtype, lens, hq, hkv, d, bs, pages)
    assert n_q * (hq // hkv) <= 16
    q = _chunk_batch(base, n_q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


@pytest.mark.parametrize("n_q", [16, 64])   # 64 rows: pipelined kernel; 256: two Q tiles
def test_warp_specialized_wait_time_out_is_reported(lib, n_q):
    # the load warp(s) announce no key tile (test hook), so the MMA and softmax waits run
    # out; the call reports PA_DEV_TIMEOUT, zeroes its outputs and leaves the context usable
    base = workloads.make_batch("wstimeout", 50, "bf16", [300], 4, 1, 64, 16, 30)
    q = _chunk_batch(base, n_q)                 # one CTA either way
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_test_set_withhold_tiles(True)
    try:
        out = _run(lib, base, q, err)
        torch.cuda.synchronize()
    finally:
        lib.pa_test_set_withhold_tiles(False)
    assert int(err.item()) == lib.PA_DEV_TIMEOUT
    assert torch.all(out == 0)
    err.zero_()
    out = _run(lib, base, q, err)               # the same call runs normally afterwards
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_attn_close(out, _ref(base, q), base.dtype)


@pytest.mark.parametrize("n_q", [40, 80])        # 160 rows: one Q tile per CTA; 320: two
def test_tensor_core_bad_seq_len_is_reported_and_zeroed(lib, n_q):
    base = workloads.make_batch("tclen", 51, "bf16", [100, 300], 32, 8, 64, 16, 40)
    q = _chunk_batch(base, n_q)
    good = base.seq_lens.clone()
    base.seq_lens[1] = base.max_blocks * base.block_size + 1   # past the table's capacity
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = _run(lib, base, q, err)
    torch.cuda.synchronize()
    assert int(err.item()) == lib.PA_DEV_BAD_SEQ_LEN
    assert torch.all(out[1] == 0)
    base.seq_lens = good
    assert_attn_close(out[:1], _ref(base, q, [0]), base.dtype)
