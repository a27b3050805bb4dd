"""Shared test helpers: tolerances, host copies of inputs, oracle slices."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# |gpu - ref| <= atol + rtol * |ref| elementwise, against the fp64 oracle
TOL = {torch.float32: 1e-5, torch.float16: 2e-2, torch.bfloat16: 2e-2}


def host_f32(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a (possibly 16-bit) tensor to a float32 numpy array."""
    return t.detach().cpu().float().numpy()


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns, for byte-exact comparisons."""
    t = t.detach().cpu().contiguous()
    view = {1: torch.int8, 2: torch.int16, 4: torch.int32}[t.element_size()]
    return t.view(view).numpy()


def assert_attn_close(got: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, what: str = ""):
    tol = TOL[dtype]
    g = got.detach().cpu().double().numpy()
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bad = err > tol + tol * np.abs(ref)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements beyond "
                           f"{tol} abs + {tol} rel; max err {err.max():.3e}")
    return float(err.max())


def oracle_seq(batch, b: int, k_pool=None, v_pool=None):
    """fp64 oracle output [Hq, d] of sequence b, reading only its own pages.

    The sequence's pages are copied to the host (device-resident pools never
    come back whole) and the block-table row is renumbered to match.
    """
    k_pool = batch.k_pool if k_pool is None else k_pool
    v_pool = batch.v_pool if v_pool is None else v_pool
    n = int(batch.seq_lens[b])
    npg = -(-n // batch.block_size)
    pages = batch.block_table[b, :npg].long().to(k_pool.device)
    ks = host_f32(k_pool.index_select(0, pages))
    vs = host_f32(v_pool.index_select(0, pages))
    q = host_f32(batch.q[b])
    return oracle.paged_decode_one(q, ks, vs, np.arange(npg), n, batch.scale, batch.block_size)


def oracle_seq_splits(batch, b: int, num_splits: int, pages_per_split: int):
    """fp64 oracle partials ([Hq, S, d], [Hq, S]) of sequence b."""
    n = int(batch.seq_lens[b])
    npg = -(-n // batch.block_size)
    pages = batch.block_table[b, :npg].long().to(batch.k_pool.device)
    ks = host_f32(batch.k_pool.index_select(0, pages))
    vs = host_f32(batch.v_pool.index_select(0, pages))
    q = host_f32(batch.q[b:b + 1])
    po, pl = oracle.splitkv_partials(q, ks, vs, np.arange(npg)[None, :], np.array([n]),
                                     batch.scale, batch.block_size, pages_per_split, num_splits)
    return po[0], pl[0]
