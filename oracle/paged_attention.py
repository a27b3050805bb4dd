"""fp64 CPU oracle for paged decode attention (test infrastructure only).

This module is the plain definition of what the paged read computes, in
NumPy float64, with no blocking, fusion or reordering beyond that
definition.  It is imported only by tests, the smoke check and the bench's
CPU-baseline leg; the CUDA library never calls it.

What it follows:

* Attention itself: softmax(Q K^T / sqrt(d)) V ("Three Attention Kernels",
  section "What is attention, really?").  ``scale`` is passed explicitly.
* Reading through a block table: the page of token p of sequence b is
  ``block_table[b][p // page_size]`` and the token sits at slot
  ``p % page_size`` of that page ("Three Attention Kernels", section
  "3. Paged KV-cache attention").
* The gather form: rebuild the contiguous history through the block table,
  then run ordinary attention over it (nanoserve "Day 20: the number the
  Triton kernel has to beat", section "What I added today": the Day-16
  gather read, the oracle the kernel is held to).
* Split-KV partials and their combine: every split reduces its own slice of
  the history to an output and a log-sum-exp; the combine takes the max
  lse, weights each split by exp(lse - max) and normalises by the sum of
  weights ("Three Attention Kernels", section "2. Split-KV
  flash-decoding").
* Cache append: "grow the table, scatter the K/V" (nanoserve Day 20,
  section "What I learned"); the table is grown by the caller, the scatter
  writes each new token's K and V rows into its page slot.
* Chunked multi-query read: nanoserve "Day 23: the real triton.jit
  paged-attention kernel" (section "What I added today") gives every query
  position i of a chunk its own program and a causal offset ``past``: query
  i sits at position past + i and sees tokens 0 .. past + i.

Readings where the pages are silent:

* Pool layout [num_pages][page_size][num_kv_heads][head_dim] (page, then
  slot, then head).
* GQA: query head h reads kv head h // (Hq / Hkv) (contiguous groups).
* A sequence of length 0 attends to nothing: its output is 0 and its lse
  is -inf; a split with no tokens has lse -inf and output 0.
* A split of ``pages_per_split`` pages covers tokens
  [s * pages_per_split * page_size, min(len, (s+1) * pages_per_split * page_size)).
* In a chunk of n_q queries, seq_len counts the history and the chunk, so
  past = seq_len - n_q; a query whose position is negative sees nothing and
  its output is 0.
* A split of a chunked read covers the same fixed page run as a decode
  split; query i's share of it stops at its causal limit past + i, so a
  split that starts after that limit is empty for that query.

Its pins live in tests/test_oracle_pins.py (single-query read, splits, merge,
append), tests/test_oracle_chunk_pins.py (chunked read) and
tests/test_oracle_chunk_split_pins.py (split of a chunked read), with the
hand-worked cases under tests/golden/.
"""

from __future__ import annotations

import numpy as np


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def kv_head_of(h: int, num_q_heads: int, num_kv_heads: int) -> int:
    """GQA mapping: contiguous groups of Hq/Hkv query heads share a kv head."""
    group = num_q_heads // num_kv_heads
    return h // group


def token_address(block_table_row, p: int, page_size: int):
    """(page, slot) of token p: page from the block table, slot inside it."""
    return int(block_table_row[p // page_size]), p % page_size


def gather_history(k_pool, v_pool, block_table_row, seq_len: int, page_size: int):
    """Contiguous K and V of one sequence, rebuilt through its block table.

    Token p comes from (page, slot) = token_address(block_table_row, p).
    Returns two arrays [seq_len, num_kv_heads, head_dim] in the pool's dtype.
    """
    addr = [token_address(block_table_row, p, page_size) for p in range(seq_len)]
    pages = np.array([a[0] for a in addr], dtype=np.int64)
    slots = np.array([a[1] for a in addr], dtype=np.int64)
    return k_pool[pages, slots], v_pool[pages, slots]


def attend(q_h, k_hist, v_hist, scale: float):
    """softmax(scale * K q) V for one query vector over one history.

    q_h [d], k_hist/v_hist [n, d].  Returns (out [d], lse) in float64 where
    lse = log(sum_t exp(scale * q.k_t)).  An empty history gives (0, -inf).
    The max is subtracted before exp, which changes nothing mathematically
    and keeps exp finite.
    """
    q_h = _f64(q_h)
    k_hist = _f64(k_hist)
    v_hist = _f64(v_hist)
    d = q_h.shape[0]
    if k_hist.shape[0] == 0:
        return np.zeros(d, dtype=np.float64), -np.inf
    s = scale * (k_hist @ q_h)
    m = s.max()
    e = np.exp(s - m)
    z = e.sum()
    out = (e / z) @ v_hist
    return out, m + np.log(z)


def paged_decode_one(q_b, k_pool, v_pool, block_table_row, seq_len: int,
                     scale: float, page_size: int):
    """Attention output [Hq, d] (float64) of one sequence of the batch."""
    n_q = q_b.shape[0]
    n_kv = k_pool.shape[2]
    k_hist, v_hist = gather_history(k_pool, v_pool, block_table_row, seq_len, page_size)
    out = np.zeros((n_q, q_b.shape[1]), dtype=np.float64)
    for h in range(n_q):
        g = kv_head_of(h, n_q, n_kv)
        out[h], _ = attend(q_b[h], k_hist[:, g, :], v_hist[:, g, :], scale)
    return out


def paged_decode(q, k_pool, v_pool, block_table, seq_lens, scale: float,
                 page_size: int):
    """Decode attention for the whole batch: out [B, Hq, d] in float64.

    q [B, Hq, d]; k_pool/v_pool [num_pages, page_size, Hkv, d];
    block_table [B, max_blocks] int; seq_lens [B] int.
    """
    b_n = q.shape[0]
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(b_n):
        out[b] = paged_decode_one(q[b], k_pool, v_pool, block_table[b],
                                  int(seq_lens[b]), scale, page_size)
    return out


def split_ranges(seq_len: int, page_size: int, pages_per_split: int, num_splits: int):
    """Token range [lo, hi) of every split; empty splits have lo == hi."""
    span = pages_per_split * page_size
    out = []
    for s in range(num_splits):
        lo = min(seq_len, s * span)
        hi = min(seq_len, (s + 1) * span)
        out.append((lo, hi))
    return out


def splitkv_partials(q, k_pool, v_pool, block_table, seq_lens, scale: float,
                     page_size: int, pages_per_split: int, num_splits: int):
    """Per-split partial outputs [B, Hq, S, d] and lse [B, Hq, S] (float64).

    Split s of a sequence attends only to its own token range; its output is
    the softmax-weighted V over that range and its lse the log of the sum of
    exp(scores) over that range.
    """
    b_n, n_q, d = q.shape
    n_kv = k_pool.shape[2]
    part = np.zeros((b_n, n_q, num_splits, d), dtype=np.float64)
    lse = np.full((b_n, n_q, num_splits), -np.inf, dtype=np.float64)
    for b in range(b_n):
        n = int(seq_lens[b])
        k_hist, v_hist = gather_history(k_pool, v_pool, block_table[b], n, page_size)
        for s, (lo, hi) in enumerate(split_ranges(n, page_size, pages_per_split, num_splits)):
            for h in range(n_q):
                g = kv_head_of(h, n_q, n_kv)
                part[b, h, s], lse[b, h, s] = attend(
                    q[b, h], k_hist[lo:hi, g, :], v_hist[lo:hi, g, :], scale)
    return part, lse


def merge_partials(partial_out, partial_lse):
    """Combine split partials: out = sum_s w_s o_s / sum_s w_s, w_s = exp(lse_s - max lse).

    partial_out [..., S, d], partial_lse [..., S].  Rows whose splits are
    all empty (every lse is -inf) give 0.
    """
    po = _f64(partial_out)
    lse = _f64(partial_lse)
    out = np.zeros(po.shape[:-2] + po.shape[-1:], dtype=np.float64)
    flat_po = po.reshape(-1, po.shape[-2], po.shape[-1])
    flat_lse = lse.reshape(-1, lse.shape[-1])
    flat_out = out.reshape(-1, po.shape[-1])
    for r in range(flat_lse.shape[0]):
        row = flat_lse[r]
        m = row.max()
        if m == -np.inf:
            continue
        w = np.exp(row - m)
        flat_out[r] = (w[:, None] * flat_po[r]).sum(axis=0) / w.sum()
    return out


def cache_append(k_pool, v_pool, k_new, v_new, block_table, positions,
                 page_size: int, seq_ids=None):
    """Scatter new tokens' K/V rows into their page slots (returns new pools).

    Token i belongs to sequence seq_ids[i] (token i -> sequence i when
    seq_ids is None) and lands at position positions[i]: page
    block_table[seq][pos // page_size], slot pos % page_size.  A pure copy:
    the pools keep their dtype and every other byte.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    for i in range(k_new.shape[0]):
        b = i if seq_ids is None else int(seq_ids[i])
        page, slot = token_address(block_table[b], int(positions[i]), page_size)
        k_out[page, slot] = k_new[i]
        v_out[page, slot] = v_new[i]
    return k_out, v_out


def paged_decode_chunk(q, k_pool, v_pool, block_table, seq_lens, scale: float,
                       page_size: int):
    """Causal read of a chunk of queries per sequence: out [B, n_q, Hq, d] (float64).

    q [B, n_q, Hq, d].  Query i of sequence b sits at position
    past_b + i with past_b = seq_lens[b] - n_q, and attends to tokens
    0 .. past_b + i of the sequence (read through its block table).
    """
    b_n, n_q, n_h, d = q.shape
    n_kv = k_pool.shape[2]
    out = np.zeros(q.shape, dtype=np.float64)
    for b in range(b_n):
        n = int(seq_lens[b])
        past = n - n_q
        k_hist, v_hist = gather_history(k_pool, v_pool, block_table[b], n, page_size)
        for i in range(n_q):
            seen = past + i + 1          # tokens 0 .. past + i
            if seen <= 0:
                continue
            for h in range(n_h):
                g = kv_head_of(h, n_h, n_kv)
                out[b, i, h], _ = attend(q[b, i, h], k_hist[:seen, g, :], v_hist[:seen, g, :],
                                         scale)
    return out


def chunk_splitkv_partials(q, k_pool, v_pool, block_table, seq_lens, scale: float,
                           page_size: int, pages_per_split: int, num_splits: int):
    """Per-split partials of the chunked read: out [B, n_q, Hq, S, d], lse [B, n_q, Hq, S].

    Split s covers the tokens of split_ranges(); query i of sequence b keeps
    the part of it at or before its position past_b + i (the causal rule of
    paged_decode_chunk) and reduces that part like a decode split.  Merging
    the splits of a query with merge_partials gives paged_decode_chunk.
    """
    b_n, n_q, n_h, d = q.shape
    n_kv = k_pool.shape[2]
    part = np.zeros((b_n, n_q, n_h, num_splits, d), dtype=np.float64)
    lse = np.full((b_n, n_q, n_h, num_splits), -np.inf, dtype=np.float64)
    for b in range(b_n):
        n = int(seq_lens[b])
        past = n - n_q
        k_hist, v_hist = gather_history(k_pool, v_pool, block_table[b], n, page_size)
        ranges = split_ranges(n, page_size, pages_per_split, num_splits)
        for i in range(n_q):
            seen = max(0, past + i + 1)
            for s, (lo, hi) in enumerate(ranges):
                hi = min(hi, seen)
                if hi <= lo:
                    continue
                for h in range(n_h):
                    g = kv_head_of(h, n_h, n_kv)
                    part[b, i, h, s], lse[b, i, h, s] = attend(
                        q[b, i, h], k_hist[lo:hi, g, :], v_hist[lo:hi, g, :], scale)
    return part, lse
