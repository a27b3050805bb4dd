"""Pins of the oracle's chunked split-KV partials to things other than themselves.

Explicit per-token loops over the block table (no gather, no shared
helper), the combine of the splits against the separately pinned chunked
read, closed forms for one-token and all-masked splits, the sum of the
splits' exp(lse) against the whole range's, and planted mistakes in the
causal clip of a split.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import oracle.paged_attention as opa

from test_oracle_chunk_pins import _random

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_chunk_split.json")


def _exact(x):
    """Fixture values: numbers, or strings 'a/b', 'ln x' and '-inf' for exact values."""
    if isinstance(x, list):
        return [_exact(e) for e in x]
    if isinstance(x, str):
        if x == "-inf":
            return -math.inf
        if x.startswith("ln "):
            return math.log(Fraction(x[3:]))
        return float(Fraction(x))
    return float(x)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _brute_partials(q, k_pool, v_pool, block_table, seq_lens, scale, page_size,
                    pages_per_split, num_splits):
    b_n, n_q, nh, d = q.shape
    group = nh // k_pool.shape[2]
    span = pages_per_split * page_size
    part = np.zeros((b_n, n_q, nh, num_splits, d))
    lse = np.full((b_n, n_q, nh, num_splits), -np.inf)
    for b in range(b_n):
        n = int(seq_lens[b])
        for i in range(n_q):
            pos = n - n_q + i
            for h in range(nh):
                for s in range(num_splits):
                    sc, vs = [], []
                    for t in range(s * span, min(n, (s + 1) * span, pos + 1)):
                        page, slot = int(block_table[b][t // page_size]), t % page_size
                        kv = k_pool[page, slot, h // group]
                        sc.append(scale * sum(float(q[b, i, h, c]) * float(kv[c])
                                              for c in range(d)))
                        vs.append(v_pool[page, slot, h // group])
                    if not sc:
                        continue
                    m = max(sc)
                    w = [math.exp(x - m) for x in sc]
                    part[b, i, h, s] = sum(wt * v for wt, v in zip(w, vs)) / sum(w)
                    lse[b, i, h, s] = m + math.log(sum(w))
    return part, lse


def _case(seed=5):
    x = _random(seed, [3, 10, 17], n_q=4, nh=4, nkv=2, d=5, ps=2)
    return x


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_chunk_split(case):
    arr = lambda key: np.array(_exact(case[key]))
    part, lse = oracle.chunk_splitkv_partials(
        arr("q"), arr("k_pool"), arr("v_pool"), np.array(case["block_table"]),
        np.array(case["seq_lens"]), case["scale"], case["page_size"], case["pages_per_split"],
        case["num_splits"])
    want_lse = arr("expected_partial_lse")
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(want_lse))
    fin = np.isfinite(want_lse)
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=0, atol=1e-12)
    np.testing.assert_allclose(part, arr("expected_partial_out"), rtol=0, atol=1e-12)
    np.testing.assert_allclose(oracle.merge_partials(part, lse), arr("expected_out"), rtol=0,
                               atol=1e-12)


def test_partials_match_explicit_loops():
    x = _case()
    for pps, ns in ((1, 9), (2, 5), (3, 3), (16, 1)):
        part, lse = oracle.chunk_splitkv_partials(**x, pages_per_split=pps, num_splits=ns)
        bp, bl = _brute_partials(**x, pages_per_split=pps, num_splits=ns)
        np.testing.assert_allclose(part, bp, rtol=0, atol=1e-12)
        np.testing.assert_array_equal(np.isinf(lse), np.isinf(bl))
        fin = np.isfinite(bl)
        np.testing.assert_allclose(lse[fin], bl[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("pps", [1, 2, 3, 7, 64])
def test_merged_splits_are_the_chunked_read(pps):
    x = _random(6, [1, 5, 23, 40], n_q=6, nh=6, nkv=3, d=8, ps=4)
    ns = max(1, math.ceil(max(math.ceil(n / 4) for n in x["seq_lens"]) / pps))
    part, lse = oracle.chunk_splitkv_partials(**x, pages_per_split=pps, num_splits=ns)
    np.testing.assert_allclose(oracle.merge_partials(part, lse), oracle.paged_decode_chunk(**x),
                               rtol=0, atol=1e-12)


def test_split_lse_sum_is_the_whole_range():
    # sum_s exp(lse_s) = sum over every visible token of exp(score), per query
    x = _case(7)
    part, lse = oracle.chunk_splitkv_partials(**x, pages_per_split=1, num_splits=9)
    whole, wl = _brute_partials(**x, pages_per_split=64, num_splits=1)
    with np.errstate(divide="ignore"):
        total = np.log(np.exp(lse).sum(axis=-1))
    np.testing.assert_allclose(total, wl[..., 0], rtol=0, atol=1e-12)


def test_one_visible_token_gives_its_value_and_score():
    # sequence of 5 tokens, chunk of 2: query 0 sits at position 3.  With one
    # token per page and one page per split, split 3 holds exactly token 3.
    rng = np.random.default_rng(8)
    q = rng.standard_normal((1, 2, 2, 3))
    kp = rng.standard_normal((6, 1, 1, 3))
    vp = rng.standard_normal((6, 1, 1, 3))
    bt = np.array([[4, 0, 5, 2, 1]])
    part, lse = oracle.chunk_splitkv_partials(q, kp, vp, bt, np.array([5]), 0.7, 1, 1, 5)
    for h in range(2):
        np.testing.assert_array_equal(part[0, 0, h, 3], vp[2, 0, 0])
        assert lse[0, 0, h, 3] == pytest.approx(0.7 * float(q[0, 0, h] @ kp[2, 0, 0]), abs=1e-15)
        # token 4 is past query 0's limit: split 4 is empty for it, not for query 1
        assert lse[0, 0, h, 4] == -np.inf and not part[0, 0, h, 4].any()
        np.testing.assert_array_equal(part[0, 1, h, 4], vp[1, 0, 0])


def _partials_with(clip):
    """The oracle's partials with the causal clip of a split replaced by clip(lo, hi, seen)."""
    def fn(q, k_pool, v_pool, block_table, seq_lens, scale, page_size, pages_per_split,
           num_splits):
        b_n, n_q, n_h, d = q.shape
        part = np.zeros((b_n, n_q, n_h, num_splits, d))
        lse = np.full((b_n, n_q, n_h, num_splits), -np.inf)
        for b in range(b_n):
            n = int(seq_lens[b])
            k, v = oracle.gather_history(k_pool, v_pool, block_table[b], n, page_size)
            ranges = oracle.split_ranges(n, page_size, pages_per_split, num_splits)
            for i in range(n_q):
                seen = max(0, n - n_q + i + 1)
                for s, (lo, hi) in enumerate(ranges):
                    lo, hi = clip(lo, hi, seen)
                    if hi <= lo:
                        continue
                    for h in range(n_h):
                        g = opa.kv_head_of(h, n_h, k_pool.shape[2])
                        part[b, i, h, s], lse[b, i, h, s] = oracle.attend(
                            q[b, i, h], k[lo:hi, g], v[lo:hi, g], scale)
        return part, lse
    return fn


MUTANTS = {
    "no_causal_clip": lambda lo, hi, seen: (lo, hi),
    "clip_off_by_one": lambda lo, hi, seen: (lo, min(hi, seen - 1)),
    "clip_one_late": lambda lo, hi, seen: (lo, min(hi, seen + 1)),
    "splits_overlap": lambda lo, hi, seen: (max(0, lo - 1), min(hi, seen)),
}


def _split_pins_pass():
    try:
        for case in _golden_cases():
            test_golden_chunk_split(case)
        test_partials_match_explicit_loops()
        for pps in (1, 2, 3, 7, 64):
            test_merged_splits_are_the_chunked_read(pps)
        test_split_lse_sum_is_the_whole_range()
        test_one_visible_token_gives_its_value_and_score()
    except Exception:
        return False
    return True


def test_unmutated_split_oracle_passes():
    assert _split_pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_split_clip_mistake_is_caught(name, monkeypatch):
    monkeypatch.setattr(oracle, "chunk_splitkv_partials", _partials_with(MUTANTS[name]))
    with np.errstate(all="ignore"):
        assert not _split_pins_pass()
