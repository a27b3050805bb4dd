"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every test appends the step's new token with pa_cache_append, reads with
pa_decode (or pa_decode_splitkv + pa_merge) and compares with the oracle:
bit-exact for the append, |gpu - ref| <= tol + tol*|ref| for attention
(tol 1e-5 for fp32 caches, 2e-2 for fp16/bf16).
"""

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_attn_close, host_bits, host_f32, oracle_seq, oracle_seq_splits

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _append(lib, bt, dev_err=None):
    lib.pa_cache_append(bt.k_new, bt.v_new, bt.k_pool, bt.v_pool, bt.block_table, bt.positions,
                        dev_err=dev_err)


def _decode(lib, bt, dev_err=None):
    out = torch.empty_like(bt.q)
    lib.pa_decode(out, bt.q, bt.k_pool, bt.v_pool, bt.block_table, bt.seq_lens, bt.scale,
                  dev_err=dev_err)
    return out


def _split(lib, bt, pps, dev_err=None):
    s = lib.pa_num_splits(bt.max_blocks, pps)
    b, hq, d = bt.q.shape
    po = torch.full((b, hq, s, d), float("nan"), device=DEV)
    pl = torch.full((b, hq, s), float("nan"), device=DEV)
    lib.pa_decode_splitkv(po, pl, bt.q, bt.k_pool, bt.v_pool, bt.block_table, bt.seq_lens,
                          bt.scale, pps, dev_err=dev_err)
    out = torch.empty_like(bt.q)
    lib.pa_merge(out, po, pl)
    return po, pl, out


def _err_buf():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def _host_after_append(cpu):
    """Oracle inputs: the step's append applied on host copies of the pools."""
    k2, v2 = oracle.cache_append(host_f32(cpu.k_pool), host_f32(cpu.v_pool), host_f32(cpu.k_new),
                                 host_f32(cpu.v_new), cpu.block_table.numpy(),
                                 cpu.positions.numpy(), cpu.block_size)
    return k2, v2


SMALL = {
    "tiny": lambda: workloads.tiny(),
    "awkward": lambda: workloads.awkward(),
    "llama1b_h16": lambda: workloads.llama1b(16),
    "llama1b_h64": lambda: workloads.llama1b(64),
    "llama1b_h256": lambda: workloads.llama1b(256),
    "llama1b_h1024": lambda: workloads.llama1b(1024),
}


# ---------------------------------------------------------------- append


@pytest.mark.parametrize("name", ["tiny", "awkward", "llama1b_h256"])
def test_append_is_bit_exact(lib, name):
    cpu = SMALL[name]()
    gpu = cpu.to(DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kb, vb = host_bits(cpu.k_pool), host_bits(cpu.v_pool)
    k_ref, v_ref = oracle.cache_append(kb, vb, host_bits(cpu.k_new), host_bits(cpu.v_new),
                                       cpu.block_table.numpy(), cpu.positions.numpy(),
                                       cpu.block_size)
    assert np.array_equal(host_bits(gpu.k_pool), k_ref)
    assert np.array_equal(host_bits(gpu.v_pool), v_ref)


def test_append_with_seq_ids_and_many_tokens(lib):
    # several tokens of several sequences in one call (a prefill-style write)
    cpu = workloads.awkward()
    gpu = cpu.to(DEV)
    g = torch.Generator().manual_seed(5)
    seq_ids, positions = [], []
    for b, n in enumerate(cpu.lens_list()):
        for p in torch.randperm(n, generator=g)[:5].tolist():
            seq_ids.append(b)
            positions.append(p)
    t = len(seq_ids)
    kn = torch.randn((t,) + cpu.k_new.shape[1:], generator=g).to(cpu.dtype)
    vn = torch.randn((t,) + cpu.k_new.shape[1:], generator=g).to(cpu.dtype)
    sid = torch.tensor(seq_ids, dtype=torch.int32)
    pos = torch.tensor(positions, dtype=torch.int32)
    err = _err_buf()
    lib.pa_cache_append(kn.to(DEV), vn.to(DEV), gpu.k_pool, gpu.v_pool, gpu.block_table,
                        pos.to(DEV), seq_ids=sid.to(DEV), dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k_ref, v_ref = oracle.cache_append(host_bits(cpu.k_pool), host_bits(cpu.v_pool),
                                       host_bits(kn), host_bits(vn), cpu.block_table.numpy(),
                                       pos.numpy(), cpu.block_size, seq_ids=sid.numpy())
    assert np.array_equal(host_bits(gpu.k_pool), k_ref)
    assert np.array_equal(host_bits(gpu.v_pool), v_ref)


# ---------------------------------------------------------------- decode


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_matches_oracle(lib, name):
    cpu = SMALL[name]()
    gpu = cpu.to(DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    out = _decode(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k2, v2 = _host_after_append(cpu)
    ref = oracle.paged_decode(host_f32(cpu.q), k2, v2, cpu.block_table.numpy(),
                              cpu.seq_lens.numpy(), cpu.scale, cpu.block_size)
    assert_attn_close(out, ref, cpu.dtype, name)


def test_decode_llama1b_h4096_full_batch(lib):
    # the benchmarked launch, every sequence: batch 64 at history 4096, 20,000-page pool
    cpu = workloads.llama1b(4096)
    gpu = cpu.to(DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    out = _decode(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for b in range(gpu.num_seqs):
        assert_attn_close(out[b], oracle_seq(gpu, b), cpu.dtype, f"seq {b}")


@pytest.mark.parametrize("name", ["tiny", "awkward", "llama1b_h256"])
def test_one_token_history_returns_v_bit_exact(lib, name):
    cpu = SMALL[name]()
    cpu.seq_lens[:] = 1
    cpu.positions[:] = 0
    gpu = cpu.to(DEV)
    _append(lib, gpu)
    out = _decode(lib, gpu)
    torch.cuda.synchronize()
    g = cpu.num_q_heads // cpu.num_kv_heads
    want = cpu.v_new.repeat_interleave(g, dim=1)          # [B, Hq, d]: v of the only token
    assert torch.equal(out.cpu(), want)


def test_page_permutation_gives_bit_identical_output(lib):
    cpu = workloads.llama1b(256, batch=16, num_pages=2000)
    gpu = cpu.to(DEV)
    out = _decode(lib, gpu)
    perm = torch.randperm(cpu.num_pages, generator=torch.Generator().manual_seed(9))
    kp = torch.empty_like(cpu.k_pool)
    vp = torch.empty_like(cpu.v_pool)
    kp[perm] = cpu.k_pool
    vp[perm] = cpu.v_pool
    bt = torch.where(cpu.block_table >= 0, perm.to(torch.int32)[cpu.block_table.clamp(min=0).long()],
                     cpu.block_table)
    gpu2 = gpu.to(DEV)
    gpu2.k_pool, gpu2.v_pool, gpu2.block_table = kp.to(DEV), vp.to(DEV), bt.to(DEV)
    out2 = _decode(lib, gpu2)
    assert torch.equal(out, out2)


def test_identical_queries_in_a_group_give_identical_outputs(lib):
    cpu = workloads.llama1b(1024, batch=4)
    cpu.q[:, 1:4] = cpu.q[:, 0:1]
    gpu = cpu.to(DEV)
    out = _decode(lib, gpu).cpu()
    for h in (1, 2, 3):
        assert torch.equal(out[:, h], out[:, 0])
    assert not torch.equal(out[:, 4], out[:, 0])


def test_zero_length_sequence_gives_zero(lib):
    cpu = workloads.awkward()
    cpu.seq_lens[2] = 0
    gpu = cpu.to(DEV)
    err = _err_buf()
    out = _decode(lib, gpu, err)
    po, pl, merged = _split(lib, gpu, 2, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.all(out[2] == 0) and torch.all(merged[2] == 0)
    assert torch.all(torch.isneginf(pl[2])) and torch.all(po[2] == 0)
    ref = oracle.paged_decode(host_f32(cpu.q), host_f32(cpu.k_pool), host_f32(cpu.v_pool),
                              cpu.block_table.numpy(), cpu.seq_lens.numpy(), cpu.scale,
                              cpu.block_size)
    assert_attn_close(out, ref, cpu.dtype)


@pytest.mark.parametrize("dtype,hq,hkv,d,bs", [
    # CUDA-core read
    ("f32", 8, 8, 256, 16),     # two chunks per lane, group 1
    ("f16", 6, 3, 16, 64),      # tiny rows (two chunks), group 2, big pages
    ("f32", 4, 1, 48, 8),       # group 4, 12 chunks per row
    ("bf16", 8, 4, 80, 16),     # head_dim outside the tensor-core list
    ("f32", 16, 2, 64, 16),     # group 8
    # tensor-core read
    ("bf16", 16, 2, 128, 1),    # one token per page, group 8
    ("bf16", 40, 8, 96, 32),    # group 5
    ("f16", 48, 4, 64, 16),     # group 12: two head tiles
    ("bf16", 32, 2, 128, 8),    # group 16, pages smaller than a tile
    ("bf16", 4, 4, 32, 4),      # group 1
    ("f16", 8, 2, 256, 16),     # widest rows
    ("bf16", 6, 2, 48, 2),      # group 3, head_dim 48
])
def test_decode_other_shapes(lib, dtype, hq, hkv, d, bs):
    lens = [1, bs - 1 if bs > 1 else 2, 3 * bs + 5, 700]
    pages = sum(-(-n // bs) for n in lens) + 7
    cpu = workloads.make_batch("shape", 21, dtype, lens, hq, hkv, d, bs, pages)
    gpu = cpu.to(DEV)
    out = _decode(lib, gpu)
    _, _, merged = _split(lib, gpu, 3)
    ref = oracle.paged_decode(host_f32(cpu.q), host_f32(cpu.k_pool), host_f32(cpu.v_pool),
                              cpu.block_table.numpy(), cpu.seq_lens.numpy(), cpu.scale, bs)
    assert_attn_close(out, ref, cpu.dtype, "decode")
    assert_attn_close(merged, ref, cpu.dtype, "split+merge")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (16, 2, 128), (8, 8, 256), (12, 4, 36)])
def test_f32_cache_at_batch_size(lib, hq, hkv, d):
    # the fp32 read (CUDA cores) on 64 ragged sequences up to 1100 tokens, every sequence
    # against the oracle, single pass and split into 7-page runs + merge
    gen = torch.Generator().manual_seed(d)
    lens = [1, 15, 16, 17] + torch.randint(1, 1101, (60,), generator=gen).tolist()
    pages = sum(-(-n // 16) for n in lens) + 9
    cpu = workloads.make_batch("f32_batch", 23, "f32", lens, hq, hkv, d, 16, pages)
    gpu = cpu.to(DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    out = _decode(lib, gpu, err)
    _, _, merged = _split(lib, gpu, 7, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k2, v2 = _host_after_append(cpu)
    ref = oracle.paged_decode(host_f32(cpu.q), k2, v2, cpu.block_table.numpy(),
                              cpu.seq_lens.numpy(), cpu.scale, 16)
    assert_attn_close(out, ref, cpu.dtype, "single pass")
    assert_attn_close(merged, ref, cpu.dtype, "split + merge")


def test_f32_bad_page_is_reported_and_zeroed(lib):
    cpu = workloads.make_batch("f32_bad", 24, "f32", [40, 300, 129], 8, 2, 64, 16, 40)
    cpu.block_table[1, 7] = cpu.num_pages + 3
    gpu = cpu.to(DEV)
    err = _err_buf()
    out = _decode(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[1] == 0)
    ref = oracle.paged_decode(host_f32(cpu.q[[0, 2]]), host_f32(cpu.k_pool), host_f32(cpu.v_pool),
                              cpu.block_table[[0, 2]].numpy(), cpu.seq_lens[[0, 2]].numpy(),
                              cpu.scale, 16)
    assert_attn_close(out[[0, 2]], ref, cpu.dtype)


# ---------------------------------------------------------------- split-KV + merge


@pytest.mark.parametrize("name,pps", [("awkward", 1), ("awkward", 3), ("tiny", 2),
                                      ("llama1b_h1024", 16), ("llama1b_h256", 64)])
def test_splitkv_partials_and_merge_match_oracle(lib, name, pps):
    cpu = SMALL[name]()
    gpu = cpu.to(DEV)
    _append(lib, gpu)
    err = _err_buf()
    po, pl, out = _split(lib, gpu, pps, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    k2, v2 = _host_after_append(cpu)
    s = po.shape[2]
    ref_po, ref_pl = oracle.splitkv_partials(host_f32(cpu.q), k2, v2, cpu.block_table.numpy(),
                                             cpu.seq_lens.numpy(), cpu.scale, cpu.block_size,
                                             pps, s)
    tol = 1e-5 if cpu.dtype == torch.float32 else 2e-2
    got_pl = pl.cpu().double().numpy()
    assert np.array_equal(np.isneginf(got_pl), np.isneginf(ref_pl))
    fin = np.isfinite(ref_pl)
    assert np.all(np.abs(got_pl[fin] - ref_pl[fin]) <= tol + tol * np.abs(ref_pl[fin]))
    assert_attn_close(po, ref_po, cpu.dtype, "partial_out")
    ref = oracle.paged_decode(host_f32(cpu.q), k2, v2, cpu.block_table.numpy(),
                              cpu.seq_lens.numpy(), cpu.scale, cpu.block_size)
    assert_attn_close(out, ref, cpu.dtype, "merged")
    # and split + merge agrees with the single-pass read
    assert_attn_close(out, _decode(lib, gpu).cpu().double().numpy(), cpu.dtype, "vs no-split")


@pytest.mark.parametrize("history", workloads.LONGCTX_HISTORIES)
def test_longctx_splitkv_full_size_sampled(lib, history):
    # batch 8, 64-page splits, 1% of keys x8; inputs drawn on the device
    gpu = workloads.longctx(history, device=DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    po, pl, out = _split(lib, gpu, gpu.pages_per_split, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert gpu.meta["n_peaky"] > 0
    # every sequence at 32K; two of the eight at 128K (the oracle's fp64 gather of one
    # 128K sequence is 2 GB)
    for b in (range(gpu.num_seqs) if history <= 32768 else (0, 5)):
        assert_attn_close(out[b], oracle_seq(gpu, b), gpu.dtype, f"seq {b}")
    ref_po, ref_pl = oracle_seq_splits(gpu, 7, po.shape[2], gpu.pages_per_split)
    assert_attn_close(po[7], ref_po, gpu.dtype, "partials seq 7")
    got = pl[7].cpu().double().numpy()
    assert np.all(np.abs(got - ref_pl) <= 2e-2 + 2e-2 * np.abs(ref_pl))
    del po, pl, out, gpu
    torch.cuda.empty_cache()


def test_ragged8b_full_size_sampled(lib):
    # batch 256, histories U[16, 8192], 160,000-page pool drawn on the device
    gpu = workloads.ragged8b(device=DEV)
    err = _err_buf()
    _append(lib, gpu, err)
    out = _decode(lib, gpu, err)
    _, _, merged = _split(lib, gpu, 64, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    lens = gpu.lens_list()
    # the 4 longest, the 4 shortest and every 10th sequence: 34 of 256
    order = np.argsort(lens)
    picks = sorted({int(x) for x in order[:4]} | {int(x) for x in order[-4:]} |
                   set(range(0, 256, 10)))
    assert len(picks) >= 32
    for b in picks:
        ref = oracle_seq(gpu, b)
        assert_attn_close(out[b], ref, gpu.dtype, f"seq {b} len {lens[b]}")
        assert_attn_close(merged[b], ref, gpu.dtype, f"split seq {b}")
    del out, merged, gpu
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- device-side errors


def test_bad_page_id_is_reported_and_zeroed(lib):
    cpu = workloads.awkward()
    cpu.block_table[3, 2] = cpu.num_pages + 5           # sequence 3 (257 tokens) points outside
    gpu = cpu.to(DEV)
    err = _err_buf()
    out = _decode(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.all(out[3] == 0)
    ref = oracle.paged_decode(host_f32(cpu.q[:3]), host_f32(cpu.k_pool), host_f32(cpu.v_pool),
                              cpu.block_table[:3].numpy(), cpu.seq_lens[:3].numpy(), cpu.scale,
                              cpu.block_size)
    assert_attn_close(out[:3], ref, cpu.dtype, "untouched sequences")
    err.zero_()
    po, pl, _ = _split(lib, gpu, 1, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert torch.isneginf(pl[3, :, 2]).all() and torch.all(po[3, :, 2] == 0)


def test_bad_seq_len_is_reported(lib):
    cpu = workloads.awkward()
    cpu.seq_lens[1] = cpu.max_blocks * cpu.block_size + 1
    gpu = cpu.to(DEV)
    err = _err_buf()
    out = _decode(lib, gpu, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 3
    assert torch.all(out[1] == 0)


@pytest.mark.parametrize("what,code", [("position", 2), ("seq_id", 4), ("page", 1)])
def test_bad_append_is_reported_and_skipped(lib, what, code):
    cpu = workloads.awkward()
    gpu = cpu.to(DEV)
    before_k = gpu.k_pool.clone()
    pos = gpu.positions.clone()
    sid = torch.arange(cpu.num_seqs, dtype=torch.int32, device=DEV)
    if what == "position":
        pos[0] = cpu.max_blocks * cpu.block_size
    elif what == "seq_id":
        sid[0] = cpu.num_seqs
    else:
        gpu.block_table[0, 0] = -3
    err = _err_buf()
    lib.pa_cache_append(gpu.k_new, gpu.v_new, gpu.k_pool, gpu.v_pool, gpu.block_table, pos,
                        seq_ids=sid, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == code
    # token 0 was skipped; the other tokens landed
    k_ref, _ = oracle.cache_append(host_bits(before_k), host_bits(before_k),
                                   host_bits(cpu.k_new[1:]), host_bits(cpu.k_new[1:]),
                                   cpu.block_table.numpy(), cpu.positions.numpy()[1:],
                                   cpu.block_size, seq_ids=np.arange(1, cpu.num_seqs))
    assert np.array_equal(host_bits(gpu.k_pool), k_ref)
