"""Pins of the fp64 oracle to things other than itself.

Each test checks the oracle against something the pages or the mathematics
fix independently of its code: hand-worked values (tests/golden), explicit
per-token loops, PyTorch's own attention routine on the gathered tensors,
closed forms, invariants and SciPy's logsumexp.  The planted-mistake tests
at the end swap one plausible bug into the oracle and check that at least
one pin catches it.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.paged_attention as opa
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _np(t):
    return t.float().numpy() if t.dtype != torch.float32 else t.numpy()


def _batch_np(bt):
    return dict(q=_np(bt.q), k_pool=_np(bt.k_pool), v_pool=_np(bt.v_pool),
                block_table=bt.block_table.numpy(), seq_lens=bt.seq_lens.numpy(),
                scale=bt.scale, page_size=bt.block_size)


def _golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def _arr(x):
    return np.array(x, dtype=np.float64)


def _lse_arr(x):
    return np.array([[[-np.inf if v == "-inf" else v for v in row] for row in b] for b in x])


# --------------------------------------------------------------------------
# hand-worked values


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_hand_worked(case):
    q = _arr(case["q"])
    kp, vp = _arr(case["k_pool"]), _arr(case["v_pool"])
    bt = np.array(case["block_table"])
    lens = np.array(case["seq_lens"])
    out = oracle.paged_decode(q, kp, vp, bt, lens, case["scale"], case["page_size"])
    np.testing.assert_allclose(out, _arr(case["expected_out"]), rtol=0, atol=1e-12)
    if "expected_lse" in case:
        _, lse = oracle.attend(q[0, 0], *[x[:, 0, :] for x in oracle.gather_history(
            kp, vp, bt[0], int(lens[0]), case["page_size"])], case["scale"])
        assert abs(lse - case["expected_lse"][0][0]) < 1e-12
    if "expected_partial_out" in case:
        po, pl = oracle.splitkv_partials(q, kp, vp, bt, lens, case["scale"], case["page_size"],
                                         case["pages_per_split"], case["num_splits"])
        np.testing.assert_allclose(po, _arr(case["expected_partial_out"]), rtol=0, atol=1e-12)
        exp_lse = _lse_arr(case["expected_partial_lse"])
        assert np.array_equal(np.isinf(pl), np.isinf(exp_lse))
        fin = np.isfinite(exp_lse)
        np.testing.assert_allclose(pl[fin], exp_lse[fin], rtol=0, atol=1e-12)
        np.testing.assert_allclose(oracle.merge_partials(po, pl), _arr(case["expected_out"]),
                                   rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# brute force: explicit per-token loops written independently of the oracle


def _brute_force(q, k_pool, v_pool, block_table, seq_lens, scale, page_size):
    b_n, n_q, d = q.shape
    n_kv = k_pool.shape[2]
    group = n_q // n_kv
    out = np.zeros((b_n, n_q, d))
    for b in range(b_n):
        n = int(seq_lens[b])
        for h in range(n_q):
            g = h // group
            scores = []
            for t in range(n):
                page = int(block_table[b][t // page_size])
                slot = t % page_size
                dot = 0.0
                for c in range(d):
                    dot += float(q[b, h, c]) * float(k_pool[page, slot, g, c])
                scores.append(scale * dot)
            if n == 0:
                continue
            m = max(scores)
            w = [math.exp(s - m) for s in scores]
            z = sum(w)
            for t in range(n):
                page = int(block_table[b][t // page_size])
                slot = t % page_size
                for c in range(d):
                    out[b, h, c] += w[t] / z * float(v_pool[page, slot, g, c])
    return out


def _small_random(seed, lens, n_q=4, n_kv=2, d=8, page_size=4, num_pages=None):
    rng = np.random.default_rng(seed)
    need = [math.ceil(n / page_size) for n in lens]
    num_pages = num_pages or sum(need) + 3
    perm = rng.permutation(num_pages)
    mb = max(1, max(need))
    bt = np.full((len(lens), mb), -1, dtype=np.int64)
    off = 0
    for i, n in enumerate(need):
        bt[i, :n] = perm[off:off + n]
        off += n
    q = rng.standard_normal((len(lens), n_q, d))
    kp = rng.standard_normal((num_pages, page_size, n_kv, d))
    vp = rng.standard_normal((num_pages, page_size, n_kv, d))
    return dict(q=q, k_pool=kp, v_pool=vp, block_table=bt,
                seq_lens=np.array(lens), scale=1 / math.sqrt(d), page_size=page_size)


def test_brute_force_small_random():
    x = _small_random(7, [1, 3, 4, 9, 17], n_q=6, n_kv=2, d=5, page_size=4)
    np.testing.assert_allclose(oracle.paged_decode(**x), _brute_force(**x), rtol=0, atol=1e-12)


def test_brute_force_tiny_config():
    x = _batch_np(workloads.tiny())
    np.testing.assert_allclose(oracle.paged_decode(**x), _brute_force(**x), rtol=0, atol=1e-12)


def test_brute_force_awkward_config():
    x = _batch_np(workloads.awkward())
    np.testing.assert_allclose(oracle.paged_decode(**x), _brute_force(**x), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# PyTorch's attention routine on independently gathered dense tensors


def _sdpa_reference(x):
    q = torch.from_numpy(np.asarray(x["q"], dtype=np.float64))
    kp = torch.from_numpy(np.asarray(x["k_pool"], dtype=np.float64))
    vp = torch.from_numpy(np.asarray(x["v_pool"], dtype=np.float64))
    bt = torch.from_numpy(np.asarray(x["block_table"], dtype=np.int64))
    ps = x["page_size"]
    n_q, n_kv = q.shape[1], kp.shape[2]
    out = torch.zeros_like(q)
    for b, n in enumerate(np.asarray(x["seq_lens"]).tolist()):
        if n == 0:
            continue
        t = torch.arange(n)
        flat_rows = bt[b, t // ps] * ps + t % ps                      # row in [P*ps]
        k = kp.reshape(-1, n_kv, kp.shape[3]).index_select(0, flat_rows)  # [n, Hkv, d]
        v = vp.reshape(-1, n_kv, vp.shape[3]).index_select(0, flat_rows)
        k = k.permute(1, 0, 2).repeat_interleave(n_q // n_kv, dim=0)  # [Hq, n, d]
        v = v.permute(1, 0, 2).repeat_interleave(n_q // n_kv, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].unsqueeze(1), k, v, scale=x["scale"])
        out[b] = o.squeeze(1)
    return out.numpy()


@pytest.mark.parametrize("maker", ["tiny", "awkward", "random"])
def test_matches_torch_sdpa(maker):
    if maker == "random":
        x = _small_random(11, [5, 16, 31, 64, 65], n_q=8, n_kv=8, d=16, page_size=8)
    else:
        x = _batch_np(getattr(workloads, maker)())
    np.testing.assert_allclose(oracle.paged_decode(**x), _sdpa_reference(x), rtol=0, atol=1e-12)


def test_matches_torch_sdpa_llama1b_slice():
    bt = workloads.llama1b(256, batch=3)
    x = _batch_np(bt)
    np.testing.assert_allclose(oracle.paged_decode(**x), _sdpa_reference(x), rtol=0, atol=1e-11)


# --------------------------------------------------------------------------
# closed forms


def test_identical_keys_give_mean_of_values():
    x = _small_random(3, [13], n_q=4, n_kv=2, d=6, page_size=4)
    x["k_pool"][:] = x["k_pool"][0, 0]
    out = oracle.paged_decode(**x)
    k, v = oracle.gather_history(x["k_pool"], x["v_pool"], x["block_table"][0], 13, 4)
    for h in range(4):
        np.testing.assert_allclose(out[0, h], v[:, h // 2, :].mean(axis=0), rtol=0, atol=1e-13)


@pytest.mark.parametrize("what", ["q_zero", "scale_zero"])
def test_flat_scores_give_mean_of_values(what):
    x = _small_random(4, [1, 7, 12], n_q=6, n_kv=3, d=4, page_size=2)
    if what == "q_zero":
        x["q"][:] = 0.0
    else:
        x["scale"] = 0.0
    out = oracle.paged_decode(**x)
    for b, n in enumerate([1, 7, 12]):
        _, v = oracle.gather_history(x["k_pool"], x["v_pool"], x["block_table"][b], n, 2)
        for h in range(6):
            np.testing.assert_allclose(out[b, h], v[:, h // 2].mean(axis=0), rtol=0, atol=1e-13)


def test_one_token_history_returns_v_exactly():
    x = _small_random(5, [1, 1, 1], n_q=4, n_kv=4, d=8, page_size=3)
    out = oracle.paged_decode(**x)
    for b in range(3):
        page = x["block_table"][b][0]
        assert np.array_equal(out[b], x["v_pool"][page, 0])


def test_empty_history_gives_zero_and_neg_inf_lse():
    x = _small_random(6, [0, 5], n_q=2, n_kv=1, d=4, page_size=4)
    out = oracle.paged_decode(**x)
    assert np.all(out[0] == 0.0)
    _, lse = oracle.attend(x["q"][0, 0], np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    assert lse == -np.inf


def test_lse_matches_scipy_logsumexp():
    from scipy.special import logsumexp
    x = _small_random(8, [37], n_q=2, n_kv=1, d=8, page_size=4)
    k, v = oracle.gather_history(x["k_pool"], x["v_pool"], x["block_table"][0], 37, 4)
    _, lse = oracle.attend(x["q"][0, 1], k[:, 0], v[:, 0], x["scale"])
    s = x["scale"] * (k[:, 0] @ x["q"][0, 1])
    assert abs(lse - logsumexp(s)) < 1e-12


def test_large_scores_stay_finite():
    # scores around 5000 overflow exp() without the max shift; softmax is shift-invariant
    x = _small_random(9, [10], n_q=1, n_kv=1, d=4, page_size=4)
    base = oracle.paged_decode(**x)
    x2 = dict(x)
    x2["q"] = x["q"].copy()
    x2["k_pool"] = x["k_pool"].copy()
    # add a component that contributes the same +5000 to every score
    x2["q"] = np.concatenate([x["q"], np.full((1, 1, 1), 1.0)], axis=2)
    x2["k_pool"] = np.concatenate([x["k_pool"], np.full(x["k_pool"].shape[:3] + (1,), 5000.0 / x["scale"])], axis=3)
    x2["v_pool"] = np.concatenate([x["v_pool"], np.zeros(x["v_pool"].shape[:3] + (1,))], axis=3)
    out = oracle.paged_decode(**x2)
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(out[..., :4], base, rtol=0, atol=1e-9)


def test_peaky_key_dominates_within_the_softmax_bound():
    # one key row scaled x8 (the long-context workload's peaky keys): when its score leads
    # every other by delta, the output is v of that token up to the weight the rest keep,
    #   |out - v_top| <= r * max_t |v_t - v_top| / (1 + r),  r = (n - 1) exp(-delta)
    rng = np.random.default_rng(31)
    n, d, ps = 40, 16, 4
    k = rng.standard_normal((n // ps, ps, 1, d)) * 0.3
    v = rng.standard_normal((n // ps, ps, 1, d))
    q = rng.standard_normal((1, 1, d))
    top = 23                                     # token 23: page 5, slot 3 (identity table)
    k[top // ps, top % ps, 0] = 8.0 * q[0, 0] / np.linalg.norm(q[0, 0])
    bt = np.arange(n // ps)[None, :]
    scale = 1.0 / math.sqrt(d)
    out = oracle.paged_decode(q, k, v, bt, np.array([n]), scale, ps)[0, 0]
    kh = k.reshape(n, d)
    vh = v.reshape(n, d)
    s = scale * (kh @ q[0, 0])
    delta = s[top] - np.max(np.delete(s, top))
    assert delta > 1.0                           # the scaled key does lead
    r = (n - 1) * math.exp(-delta)
    bound = r * np.max(np.abs(vh - vh[top])) / (1 + r)
    assert np.max(np.abs(out - vh[top])) <= bound + 1e-12
    # and it is no closed form by accident: the other tokens still move the output
    assert np.max(np.abs(out - vh[top])) > 0


# --------------------------------------------------------------------------
# invariants


def test_page_permutation_invariance():
    x = _small_random(12, [9, 30, 4], n_q=4, n_kv=2, d=6, page_size=4, num_pages=20)
    base = oracle.paged_decode(**x)
    rng = np.random.default_rng(0)
    perm = rng.permutation(20)          # new position of old page p is perm[p]
    kp = np.empty_like(x["k_pool"])
    vp = np.empty_like(x["v_pool"])
    kp[perm] = x["k_pool"]
    vp[perm] = x["v_pool"]
    bt = np.where(x["block_table"] >= 0, perm[np.maximum(x["block_table"], 0)], -1)
    out = oracle.paged_decode(**{**x, "k_pool": kp, "v_pool": vp, "block_table": bt})
    assert np.array_equal(out, base)


def test_gqa_identical_queries_give_identical_outputs():
    x = _small_random(13, [21], n_q=8, n_kv=2, d=4, page_size=4)
    x["q"][0, 1:4] = x["q"][0, 0]
    x["q"][0, 5:8] = x["q"][0, 4]
    out = oracle.paged_decode(**x)
    for h in (1, 2, 3):
        assert np.array_equal(out[0, h], out[0, 0])
    for h in (5, 6, 7):
        assert np.array_equal(out[0, h], out[0, 4])
    assert not np.allclose(out[0, 0], out[0, 4])


def test_gqa_mapping_contiguous_groups():
    # V of kv head g is the constant g: head h must read back exactly h // (Hq/Hkv)
    x = _small_random(14, [6, 11], n_q=12, n_kv=4, d=3, page_size=4)
    for g in range(4):
        x["v_pool"][:, :, g, :] = float(g)
    out = oracle.paged_decode(**x)
    for h in range(12):
        np.testing.assert_allclose(out[:, h, :], h // 3, rtol=0, atol=1e-14)


@pytest.mark.parametrize("pps,lens", [(1, [1, 5, 9]), (2, [16, 17, 33]), (3, [48, 3, 100])])
def test_split_then_merge_equals_no_split(pps, lens):
    x = _small_random(15, lens, n_q=4, n_kv=2, d=6, page_size=4)
    mb = x["block_table"].shape[1]
    s = -(-mb // pps)
    po, pl = oracle.splitkv_partials(**x, pages_per_split=pps, num_splits=s)
    np.testing.assert_allclose(oracle.merge_partials(po, pl), oracle.paged_decode(**x),
                               rtol=0, atol=1e-12)


def test_merge_special_cases():
    rng = np.random.default_rng(1)
    po = rng.standard_normal((3, 1, 5))
    # a single split is returned unchanged
    np.testing.assert_allclose(oracle.merge_partials(po, np.array([[0.7], [-3.0], [40.0]])),
                               po[:, 0, :], rtol=0, atol=1e-15)
    # all splits empty -> 0
    po2 = rng.standard_normal((2, 4, 5))
    out = oracle.merge_partials(po2, np.full((2, 4), -np.inf))
    assert np.all(out == 0.0)
    # equal lse -> plain average; an empty split carries no weight
    lse = np.array([[1.5, 1.5, -np.inf, 1.5]])
    np.testing.assert_allclose(oracle.merge_partials(po2[:1], lse)[0],
                               po2[0, [0, 1, 3]].mean(axis=0), rtol=0, atol=1e-14)


def test_append_then_gather_is_byte_equal():
    bt = workloads.awkward()
    x = _batch_np(bt)
    kp16, vp16 = bt.k_pool.numpy(), bt.v_pool.numpy()
    k2, v2 = oracle.cache_append(kp16, vp16, bt.k_new.numpy(), bt.v_new.numpy(),
                                 bt.block_table.numpy(), bt.positions.numpy(), bt.block_size)
    assert k2.dtype == np.float16
    for b, n in enumerate(bt.lens_list()):
        k, v = oracle.gather_history(k2, v2, x["block_table"][b], n, bt.block_size)
        assert k[n - 1].tobytes() == bt.k_new[b].numpy().tobytes()
        assert v[n - 1].tobytes() == bt.v_new[b].numpy().tobytes()
        # the rest of the history is untouched
        k0, _ = oracle.gather_history(kp16, vp16, x["block_table"][b], n, bt.block_size)
        assert k[:n - 1].tobytes() == k0[:n - 1].tobytes()
    # exactly B rows changed in each pool
    changed = (k2 != kp16).any(axis=(2, 3)).sum()
    assert changed <= bt.num_seqs


def test_append_with_seq_ids_lands_in_the_right_table_row():
    rng = np.random.default_rng(2)
    kp = rng.standard_normal((6, 2, 1, 2))
    bt = np.array([[4, 1], [0, 5]])
    kn = np.array([[[7.0, 7.0]], [[9.0, 9.0]]])
    k2, _ = oracle.cache_append(kp, kp, kn, kn, bt, positions=[3, 0], page_size=2, seq_ids=[0, 1])
    assert np.array_equal(k2[1, 1, 0], [7.0, 7.0])   # seq 0, pos 3 -> page bt[0][1]=1, slot 1
    assert np.array_equal(k2[0, 0, 0], [9.0, 9.0])   # seq 1, pos 0 -> page bt[1][0]=0, slot 0
    k3, _ = oracle.cache_append(kp, kp, kn, kn, bt, positions=[3, 0], page_size=2, seq_ids=[1, 1])
    assert np.array_equal(k3[5, 1, 0], [7.0, 7.0])   # seq 1, pos 3 -> page 5, slot 1


# --------------------------------------------------------------------------
# planted mistakes: each one must be caught by a pin above


def _pins_pass():
    """Run a representative subset of the pins; False if any fails."""
    checks = [
        lambda: [test_golden_hand_worked(c) for c in _golden_cases()],
        test_brute_force_small_random,
        lambda: test_matches_torch_sdpa("random"),
        test_gqa_mapping_contiguous_groups,
        test_one_token_history_returns_v_exactly,
        lambda: test_split_then_merge_equals_no_split(2, [16, 17, 33]),
        test_append_with_seq_ids_lands_in_the_right_table_row,
    ]
    for c in checks:
        try:
            c()
        except Exception:  # an assertion, or a crash the mistake causes
            return False
    return True


def _attend_no_scale(q_h, k, v, scale):
    return _ORIG_ATTEND(q_h, k, v, 1.0)


def _attend_no_max_shift(q_h, k, v, scale):
    q_h, k, v = (np.asarray(a, dtype=np.float64) for a in (q_h, k, v))
    if k.shape[0] == 0:
        return np.zeros(q_h.shape[0]), -np.inf
    with np.errstate(over="ignore", invalid="ignore"):
        e = np.exp(scale * (k @ q_h))
        return (e / e.sum()) @ v, np.log(e.sum())


def _attend_transposed_pv(q_h, k, v, scale):
    q_h, k, v = (np.asarray(a, dtype=np.float64) for a in (q_h, k, v))
    if k.shape[0] == 0:
        return np.zeros(q_h.shape[0]), -np.inf
    s = scale * (k @ q_h)
    e = np.exp(s - s.max())
    p = e / e.sum()
    n, d = v.shape
    # wrong: weights applied along the channel axis of a square-cropped V
    m = min(n, d)
    out = np.zeros(d)
    out[:m] = v[:m, :m].T @ p[:m] if n >= 1 else 0
    return out, s.max() + np.log(e.sum())


def _attend_lse_without_max(q_h, k, v, scale):
    out, lse = _ORIG_ATTEND(q_h, k, v, scale)
    if k.shape[0] == 0:
        return out, lse
    s = scale * (np.asarray(k, np.float64) @ np.asarray(q_h, np.float64))
    return out, lse - s.max()


_ORIG_ATTEND = opa.attend

MUTANTS = {
    "gqa_modulo_mapping": ("kv_head_of", lambda h, nq, nkv: h % nkv),
    "slot_and_page_swapped": ("token_address", lambda row, p, ps: (int(row[p % ps]) if p % ps < len(row) else 0, p // ps)),
    "off_by_one_slot": ("token_address", lambda row, p, ps: (int(row[p // ps]), (p + 1) % ps)),
    "scale_dropped": ("attend", _attend_no_scale),
    "max_shift_dropped": ("attend", _attend_no_max_shift),
    "transposed_pv": ("attend", _attend_transposed_pv),
    "lse_missing_max": ("attend", _attend_lse_without_max),
}


def test_unmutated_oracle_passes_the_pin_subset():
    assert _pins_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(opa, attr, fn)
    with np.errstate(all="ignore"):
        assert not _pins_pass(), f"planted mistake {name} went unnoticed"
