"""The split read over a planned work list (pa_decode_work + pa_merge).

The plan comes from pa_plan_work on the host lengths; the merged output
must match the fp64 oracle, and the per-item partials the oracle's
attention over exactly the item's token range.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_attn_close, host_f32, oracle_seq

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _work(lib, g, target, minp, err=None):
    items, slots = lib.pa_plan_work(g.seq_lens.cpu(), g.num_kv_heads, g.block_size, target, minp)
    b, hq, d = g.q.shape
    po = torch.full((b, hq, slots, d), float("nan"), device=DEV)
    pl = torch.full((b, hq, slots), float("nan"), device=DEV)
    lib.pa_decode_work(po, pl, items.to(DEV), g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                       g.scale, dev_err=err)
    out = torch.empty_like(g.q)
    lib.pa_merge(out, po, pl)
    torch.cuda.synchronize()
    return items, po, pl, out


@pytest.mark.parametrize("target,minp", [(64, 1), (600, 1), (600, 4), (5000, 1)])
def test_awkward_with_an_empty_sequence(lib, target, minp):
    cpu = workloads.awkward()
    cpu.seq_lens[1] = 0
    g = cpu.to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    items, po, pl, out = _work(lib, g, target, minp, err)
    assert int(err.item()) == 0
    ref = oracle.paged_decode(host_f32(cpu.q), host_f32(cpu.k_pool), host_f32(cpu.v_pool),
                              cpu.block_table.numpy(), cpu.seq_lens.numpy(), cpu.scale,
                              cpu.block_size)
    assert_attn_close(out, ref, cpu.dtype)
    assert torch.all(out[1] == 0)
    # each item's partial is attention over exactly its token range
    q, k, v = host_f32(cpu.q), host_f32(cpu.k_pool), host_f32(cpu.v_pool)
    for s, t0, t1, w in items.tolist():
        slot, count = w & 0xFFFF, w >> 16
        kh, vh = oracle.gather_history(k, v, cpu.block_table[s].numpy(), int(cpu.seq_lens[s]), 16)
        for h in range(cpu.num_q_heads):
            gk = oracle.kv_head_of(h, cpu.num_q_heads, cpu.num_kv_heads)
            o_ref, lse_ref = oracle.attend(q[s, h], kh[t0:t1, gk], vh[t0:t1, gk], cpu.scale)
            got_l = float(pl[s, h, slot])
            if t1 == t0:
                assert got_l == float("-inf")
                continue
            assert abs(got_l - lse_ref) <= 2e-2 + 2e-2 * abs(lse_ref)
            assert_attn_close(po[s, h, slot], o_ref, cpu.dtype)
        # unused slots of the sequence are marked empty
        assert torch.isneginf(pl[s, :, count:]).all()


def test_ragged8b_full_size_sampled(lib):
    g = workloads.ragged8b(device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    items, _, _, out = _work(lib, g, 4 * 456, 16, err)
    assert int(err.item()) == 0
    assert int(items[:, 0].unique().numel()) == g.num_seqs
    lens = g.lens_list()
    # the 4 longest, the 4 shortest and every 10th sequence: 34 of 256
    order = np.argsort(lens)
    picks = sorted({int(x) for x in order[:4]} | {int(x) for x in order[-4:]} |
                   set(range(0, 256, 10)))
    for b in picks:
        assert_attn_close(out[b], oracle_seq(g, b), g.dtype, f"seq {b}")
    del g, out
    torch.cuda.empty_cache()


def test_malformed_item_is_reported(lib):
    g = workloads.awkward().to(DEV)
    items, slots = lib.pa_plan_work(g.seq_lens.cpu(), 4, 16, 64, 1)
    items[0, 0] = 99                                   # no such sequence
    po = torch.zeros((4, 12, slots, 48), device=DEV)
    pl = torch.zeros((4, 12, slots), device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_decode_work(po, pl, items.to(DEV), g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                       g.scale, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 5
