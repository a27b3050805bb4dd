"""The host work planner (pa_plan_work): no GPU involved.

Checks the plan's contract on random ragged batches: every sequence's
tokens covered exactly once by its items in slot order, near-equal item
sizes of at least the minimum, the CTA count near the target, longest
items first, and refusals for bad arguments.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_184_gb300 as pa


def _decode(items):
    it = items.numpy()
    return it[:, 0], it[:, 1], it[:, 2], it[:, 3] & 0xFFFF, it[:, 3] >> 16


@pytest.mark.parametrize("seed", range(6))
def test_plan_covers_every_sequence_once(lib, seed):
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 300))
    lens = rng.integers(0, 9000, size=b).astype(np.int32)
    lens[rng.integers(0, b)] = 0
    bs, hkv, target, minp = 16, 8, int(rng.integers(100, 4000)), int(rng.integers(1, 64))
    items, slots = lib.pa_plan_work(torch.from_numpy(lens), hkv, bs, target, minp)
    seq, t0, t1, slot, count = _decode(items)
    assert slots == count.max()
    for s in range(b):
        mine = np.nonzero(seq == s)[0]
        assert len(mine) >= 1
        order = mine[np.argsort(slot[mine])]
        assert list(slot[order]) == list(range(len(mine)))
        assert np.all(count[mine] == len(mine))
        assert t0[order[0]] == 0 and t1[order[-1]] == lens[s]
        assert np.all(t1[order[:-1]] == t0[order[1:]])
        # page-aligned cuts, near-equal sizes of at least the minimum (bar the tail)
        assert np.all(t0[order] % bs == 0)
        pages = -(-(t1[order] - t0[order]) // bs)
        if len(mine) > 1:
            assert pages.max() - pages.min() <= 1
            want = max(minp, -(-int(np.sum(-(-lens // bs))) // max(1, target // hkv)))
            assert pages.min() >= want and pages.max() < 2 * want + 1
    sizes = t1 - t0
    assert np.all(np.diff(sizes) <= 0)          # longest first
    total_pages = int(np.sum(-(-lens // bs)))
    want = max(minp, -(-total_pages // max(1, target // hkv)))
    assert len(items) <= b + total_pages // want + 1


def test_plan_balances_toward_the_target(lib):
    lens = torch.full((8,), 131072, dtype=torch.int32)
    items, slots = lib.pa_plan_work(lens, 8, 16, 8 * 456, 1)
    assert len(items) * 8 == pytest.approx(8 * 456, rel=0.02)
    assert slots == len(items) // 8


@pytest.mark.parametrize("args", [
    (0, 8, 16, 100, 1), (4, 0, 16, 100, 1), (4, 8, 0, 100, 1), (4, 8, 16, 0, 1), (4, 8, 16, 100, 0),
])
def test_plan_refuses_bad_arguments(lib, args):
    b, hkv, bs, target, minp = args
    lens = (ctypes.c_int32 * max(1, b))(*([100] * max(1, b)))
    items = (ctypes.c_int32 * 400)()
    slots = ctypes.c_int32(0)
    n = lib.raw().pa_plan_work(ctypes.addressof(lens), b, hkv, bs, target, minp,
                               ctypes.addressof(items), 100, ctypes.byref(slots))
    assert n == -1


def test_plan_refuses_a_small_buffer_and_negative_lengths(lib):
    lens = (ctypes.c_int32 * 3)(5000, 5000, -1)
    items = (ctypes.c_int32 * 8)()
    slots = ctypes.c_int32(0)
    assert lib.raw().pa_plan_work(ctypes.addressof(lens), 2, 8, 16, 10000, 1,
                                  ctypes.addressof(items), 2, ctypes.byref(slots)) == -1
    assert lib.raw().pa_plan_work(ctypes.addressof(lens), 3, 8, 16, 100, 1,
                                  ctypes.addressof(items), 2, ctypes.byref(slots)) == -1


def test_plan_fits_a_buffer_of_exactly_its_size(lib):
    lens_list = [16, 5000, 3000, 12000, 1, 700]
    lens = (ctypes.c_int32 * len(lens_list))(*lens_list)

    def plan(max_items):
        items = (ctypes.c_int32 * (4 * 1000))()
        slots = ctypes.c_int32(0)
        n = lib.raw().pa_plan_work(ctypes.addressof(lens), len(lens_list), 8, 16, 600, 1,
                                   ctypes.addressof(items), max_items, ctypes.byref(slots))
        return n, list(items)[:4 * max(n, 0)], slots.value

    n, items, slots = plan(1000)
    assert n > len(lens_list)                      # the long sequences are cut
    assert plan(n) == (n, items, slots)            # the same plan in a buffer of n items
    assert plan(n - 1)[0] == -1
