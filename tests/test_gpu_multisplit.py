"""Split-KV reads where one CTA covers several consecutive splits.

When a batch has few (sequence, kv head) pairs and many splits, the read
gives each CTA k > 1 consecutive splits so the grid fits one wave (on a
152-SM GB300 every case below except the 8-page control takes that path).
Every split's partial output and lse must still match the oracle's split
partials, a bad page must zero only the split it belongs to, and the merge
must match the single-pass oracle.
"""

import numpy as np
import pytest
import torch

import workloads
from helpers import assert_attn_close, oracle_seq, oracle_seq_splits

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _split(lib, g, pps, err=None):
    s = lib.pa_num_splits(g.max_blocks, pps)
    po = torch.full((g.num_seqs, g.num_q_heads, s, g.head_dim), float("nan"), device=DEV)
    pl = torch.full((g.num_seqs, g.num_q_heads, s), float("nan"), device=DEV)
    lib.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                          pps, dev_err=err)
    out = torch.empty_like(g.q)
    lib.pa_merge(out, po, pl)
    torch.cuda.synchronize()
    return po, pl, out


def _check_partials(g, po, pl, b, pps, skip=()):
    ref_po, ref_pl = oracle_seq_splits(g, b, po.shape[2], pps)
    keep = [s for s in range(po.shape[2]) if s not in skip]
    assert_attn_close(po[b][:, keep], ref_po[:, keep], g.dtype, f"partials seq {b}")
    got = pl[b][:, keep].double().cpu().numpy()
    ref = ref_pl[:, keep]
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    fin = np.isfinite(ref)
    assert np.all(np.abs(got[fin] - ref[fin]) <= 2e-2 + 2e-2 * np.abs(ref[fin]))


@pytest.mark.parametrize("hq,hkv,d,pps", [(8, 2, 128, 1), (8, 2, 128, 2), (8, 2, 128, 3),
                                          (16, 2, 64, 1), (8, 2, 128, 8)])
def test_many_splits_per_cta(lib, hq, hkv, d, pps):
    lens = [8192, 5000]
    g = workloads.make_batch("multi", 31, "bf16", lens, hq, hkv, d, 16, 900, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    po, pl, out = _split(lib, g, pps, err)
    assert int(err.item()) == 0
    for b in range(2):
        _check_partials(g, po, pl, b, pps)
        assert_attn_close(out[b], oracle_seq(g, b), g.dtype, f"merged seq {b}")


def test_bad_page_zeroes_only_its_split(lib):
    g = workloads.make_batch("multi_bad", 32, "bf16", [8192, 5000], 8, 2, 128, 16, 900,
                             device=DEV)
    good = g.block_table.clone()
    g.block_table[0, 100] = g.num_pages + 3
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    po, pl, _ = _split(lib, g, 1, err)
    assert int(err.item()) == 1
    assert torch.isneginf(pl[0, :, 100]).all() and torch.all(po[0, :, 100] == 0)
    g.block_table = good
    _check_partials(g, po, pl, 0, 1, skip=(100,))
    _check_partials(g, po, pl, 1, 1)
