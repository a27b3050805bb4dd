"""Pins of the oracle's chunked multi-query read to things other than itself.

Hand-worked causal cases, the reduction of a one-query chunk to the
(separately pinned) single-query read, explicit per-token loops, PyTorch's
scaled_dot_product_attention with an explicit causal mask, and planted
mistakes in the causal offset.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.paged_attention as opa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_chunk.json")


def _cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _random(seed, lens, n_q, nh=4, nkv=2, d=6, ps=4):
    rng = np.random.default_rng(seed)
    need = [math.ceil(n / ps) for n in lens]
    npg = sum(need) + 2
    perm = rng.permutation(npg)
    bt = np.full((len(lens), max(need)), -1)
    off = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[off:off + n]
        off += n
    return dict(q=rng.standard_normal((len(lens), n_q, nh, d)),
                k_pool=rng.standard_normal((npg, ps, nkv, d)),
                v_pool=rng.standard_normal((npg, ps, nkv, d)), block_table=bt,
                seq_lens=np.array(lens), scale=1 / math.sqrt(d), page_size=ps)


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_golden_chunk(case):
    out = oracle.paged_decode_chunk(np.array(case["q"]), np.array(case["k_pool"]),
                                    np.array(case["v_pool"]), np.array(case["block_table"]),
                                    np.array(case["seq_lens"]), case["scale"], case["page_size"])
    np.testing.assert_allclose(out, np.array(case["expected_out"]), rtol=0, atol=1e-12)


def test_one_query_chunk_is_the_single_query_read():
    x = _random(1, [1, 7, 20], n_q=1)
    single = dict(x, q=x["q"][:, 0])
    np.testing.assert_allclose(oracle.paged_decode_chunk(**x)[:, 0], oracle.paged_decode(**single),
                               rtol=0, atol=0)


def test_each_query_is_a_single_query_read_of_its_prefix():
    x = _random(2, [9, 17], n_q=5)
    out = oracle.paged_decode_chunk(**x)
    for i in range(5):
        lens = x["seq_lens"] - 5 + i + 1
        single = dict(x, q=x["q"][:, i], seq_lens=lens)
        np.testing.assert_allclose(out[:, i], oracle.paged_decode(**single), rtol=0, atol=1e-14)


def _brute(q, k_pool, v_pool, block_table, seq_lens, scale, page_size):
    b_n, n_q, nh, d = q.shape
    group = nh // k_pool.shape[2]
    out = np.zeros(q.shape)
    for b in range(b_n):
        for i in range(n_q):
            pos = int(seq_lens[b]) - n_q + i
            for h in range(nh):
                sc, vs = [], []
                for t in range(pos + 1):
                    page, slot = int(block_table[b][t // page_size]), t % page_size
                    kv = k_pool[page, slot, h // group]
                    sc.append(scale * sum(float(q[b, i, h, c]) * float(kv[c]) for c in range(d)))
                    vs.append(v_pool[page, slot, h // group])
                if not sc:
                    continue
                m = max(sc)
                w = [math.exp(s - m) for s in sc]
                out[b, i, h] = sum(wt * v for wt, v in zip(w, vs)) / sum(w)
    return out


def test_brute_force_loops():
    x = _random(3, [4, 11, 2], n_q=4, nh=6, nkv=3, d=5, ps=2)
    np.testing.assert_allclose(oracle.paged_decode_chunk(**x), _brute(**x), rtol=0, atol=1e-12)


def test_torch_sdpa_with_explicit_causal_mask():
    x = _random(4, [16, 33, 70], n_q=8, nh=8, nkv=2, d=16, ps=8)
    q = torch.from_numpy(x["q"])
    kp, vp = torch.from_numpy(x["k_pool"]), torch.from_numpy(x["v_pool"])
    ps, n_q = x["page_size"], 8
    out = np.zeros(x["q"].shape)
    for b, n in enumerate(x["seq_lens"].tolist()):
        t = torch.arange(n)
        rows = torch.from_numpy(x["block_table"][b])[t // ps] * ps + t % ps
        k = kp.reshape(-1, 2, 16).index_select(0, rows).permute(1, 0, 2).repeat_interleave(4, 0)
        v = vp.reshape(-1, 2, 16).index_select(0, rows).permute(1, 0, 2).repeat_interleave(4, 0)
        pos = n - n_q + torch.arange(n_q)
        mask = t[None, :] <= pos[:, None]                   # [n_q, n]: bottom-right causal
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].permute(1, 0, 2), k, v, attn_mask=mask, scale=x["scale"])
        out[b] = o.permute(1, 0, 2).numpy()
    np.testing.assert_allclose(oracle.paged_decode_chunk(**x), out, rtol=0, atol=1e-12)


def _chunk_with(seen_of):
    """The oracle's chunk read with the causal limit replaced by seen_of(n, n_q, i)."""
    def fn(q, k_pool, v_pool, block_table, seq_lens, scale, page_size):
        b_n, n_q, n_h, _ = q.shape
        out = np.zeros(q.shape)
        for b in range(b_n):
            n = int(seq_lens[b])
            k, v = oracle.gather_history(k_pool, v_pool, block_table[b], n, page_size)
            for i in range(n_q):
                seen = seen_of(n, n_q, i)
                if seen <= 0:
                    continue
                for h in range(n_h):
                    g = opa.kv_head_of(h, n_h, k_pool.shape[2])
                    out[b, i, h], _ = oracle.attend(q[b, i, h], k[:seen, g], v[:seen, g], scale)
        return out
    return fn


MUTANTS = {
    "limit_off_by_one": lambda n, nq, i: n - nq + i,
    "past_off_by_one": lambda n, nq, i: n - nq + i + 2,
    "top_left_alignment": lambda n, nq, i: i + 1,
    "no_causal_mask": lambda n, nq, i: n,
}


def _chunk_pins_pass():
    try:
        for c in _cases():
            test_golden_chunk(c)
        test_brute_force_loops()
        test_each_query_is_a_single_query_read_of_its_prefix()
        test_torch_sdpa_with_explicit_causal_mask()
    except Exception:
        return False
    return True


def test_unmutated_chunk_oracle_passes():
    assert _chunk_pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_causal_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(oracle, "paged_decode_chunk", _chunk_with(MUTANTS[name]))
    with np.errstate(all="ignore"):
        assert not _chunk_pins_pass()
