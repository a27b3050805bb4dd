"""Seeded synthetic decode-step inputs for the paged KV-cache read.

This module only draws random numbers and lays them out as a paged cache:
a fixed pool of pages, per-sequence block tables, query vectors and the
new token's K/V.  It holds none of the attention arithmetic, so both the
CUDA path and the CPU oracle can take their inputs from here.

Shapes follow the workloads the pages describe (nanoserve "Day 20: the
number the Triton kernel has to beat" uses the Llama-3.2-1B head layout;
"Three Attention Kernels", section "Benchmark method", sweeps contexts of
1K to 16K).  Named configurations:

* ``tiny``      : 1 sequence, history 64, Hq 32 / Hkv 8, d 64, fp32, pool 16.
* ``awkward``   : histories {1, 13, 100, 257}, Hq 12 / Hkv 4, d 48, fp16.
* ``llama1b``   : batch 64, one history from {16, 64, 256, 1024, 4096},
                  Hq 32 / Hkv 8, d 64, bf16, pool of 20,000 pages.
* ``ragged8b``  : batch 256, histories uniform in [16, 8192], Hq 32 / Hkv 8,
                  d 128, bf16 with std 0.5, pool of 160,000 pages.
* ``longctx``   : batch 8, history 32,768 or 131,072, Hq 32 / Hkv 8, d 128,
                  bf16, 1% of keys scaled by 8, 64-page KV splits.
* ``dense``     : a contiguous (non-paged) cache, the shape of the split-KV
                  benchmark of "Three Attention Kernels" ("Benchmark method":
                  B 4, H 16, D 64, one query, fp16, contexts 1K to 16K).  The
                  pool is the batch's K/V in order and the block table is the
                  identity, so [B][N][H][D] memory is read as pages.

Draw order is fixed: pool permutation, block tables, q, K pool, V pool,
peaky-key mask, new K, new V.  K/V pools are drawn page-chunk by page-chunk
in float32 and cast, so that a 10 GB pool never needs a float32 copy.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

# page chunk used when drawing a pool: fixed, so the stream of draws is too
_POOL_CHUNK_PAGES = 2048

DTYPES = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass
class PagedBatch:
    """One decode step over a paged cache.

    Layouts (all contiguous, row-major):
      q            [B, Hq, d]                 dtype
      k_pool/v_pool[num_pages, block_size, Hkv, d] dtype
      block_table  [B, max_blocks] int32, entries past ceil(len/bs) are -1
      seq_lens     [B] int32, tokens attended including the appended one
      k_new/v_new  [B, Hkv, d] dtype, the token appended at position len-1
      positions    [B] int32 (= seq_lens - 1)
    """

    name: str
    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    seq_lens: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    positions: torch.Tensor
    scale: float
    block_size: int
    seed: int
    pages_per_split: int = 64
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return self.q.shape[0]

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pool.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_pool.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_table.shape[1]

    @property
    def dtype(self) -> torch.dtype:
        return self.q.dtype

    def lens_list(self) -> list:
        return [int(x) for x in self.seq_lens.tolist()]

    def to(self, device) -> "PagedBatch":
        out = PagedBatch(**{**self.__dict__})
        for name in ("q", "k_pool", "v_pool", "block_table", "seq_lens",
                     "k_new", "v_new", "positions"):
            setattr(out, name, getattr(self, name).to(device))
        return out

    def kv_bytes(self) -> int:
        """Bytes of K and V the read touches: sum_b len_b * Hkv * d * 2 * elem."""
        elem = self.q.element_size()
        return sum(self.lens_list()) * self.num_kv_heads * self.head_dim * 2 * elem


def _draw_pool(gen, num_pages, block_size, hkv, d, std, dtype, device):
    pool = torch.empty((num_pages, block_size, hkv, d), dtype=dtype, device=device)
    for p0 in range(0, num_pages, _POOL_CHUNK_PAGES):
        p1 = min(num_pages, p0 + _POOL_CHUNK_PAGES)
        chunk = torch.randn((p1 - p0, block_size, hkv, d), generator=gen,
                            dtype=torch.float32, device=device)
        if std != 1.0:
            chunk.mul_(std)
        pool[p0:p1].copy_(chunk)
    return pool


def make_batch(name: str, seed: int, dtype: str, lens: Sequence[int],
               num_q_heads: int, num_kv_heads: int, head_dim: int,
               block_size: int, num_pages: int, std: float = 1.0,
               peaky_frac: float = 0.0, peaky_factor: float = 8.0,
               max_blocks: Optional[int] = None, pages_per_split: int = 64,
               device: str = "cpu", take_pages: Optional[int] = None) -> PagedBatch:
    """Draw one decode step.

    Pages are assigned without replacement: a seeded permutation of the pool
    is cut into consecutive runs, one run per sequence, so block tables are
    random and non-contiguous.  ``take_pages`` limits the permutation to its
    first entries (the tiny case takes 4 of 16 pages).
    """
    tdtype = DTYPES[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    lens = [int(x) for x in lens]
    b = len(lens)
    need = [math.ceil(n / block_size) for n in lens]
    if max_blocks is None:
        max_blocks = max(1, max(need))
    if sum(need) > num_pages:
        raise ValueError(f"{name}: {sum(need)} pages needed, pool has {num_pages}")
    # 1. pool permutation, 2. block tables
    perm = torch.randperm(num_pages, generator=gen, device=device).to(torch.int32)
    if take_pages is not None:
        perm = perm[:take_pages]
    block_table = torch.full((b, max_blocks), -1, dtype=torch.int32, device=device)
    off = 0
    for i, n in enumerate(need):
        block_table[i, :n] = perm[off:off + n]
        off += n
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=device)
    # 3. q, 4. K pool, 5. V pool
    q = (torch.randn((b, num_q_heads, head_dim), generator=gen,
                     dtype=torch.float32, device=device) * std).to(tdtype)
    k_pool = _draw_pool(gen, num_pages, block_size, num_kv_heads, head_dim, std, tdtype, device)
    v_pool = _draw_pool(gen, num_pages, block_size, num_kv_heads, head_dim, std, tdtype, device)
    # 6. peaky keys: a Bernoulli mask over (sequence, token); the whole key
    #    row (all kv heads) of a chosen token is multiplied by peaky_factor
    n_peaky = 0
    if peaky_frac > 0.0:
        for i, n in enumerate(lens):
            mask = torch.rand((n,), generator=gen, device=device) < peaky_frac
            t = torch.nonzero(mask).flatten()
            if t.numel():
                pages = block_table[i].long()[t // block_size]
                slots = t % block_size
                k_pool[pages, slots] = (k_pool[pages, slots].float() * peaky_factor).to(tdtype)
                n_peaky += int(t.numel())
    # 7. new K, 8. new V: the token each sequence appends this step
    k_new = (torch.randn((b, num_kv_heads, head_dim), generator=gen,
                         dtype=torch.float32, device=device) * std).to(tdtype)
    v_new = (torch.randn((b, num_kv_heads, head_dim), generator=gen,
                         dtype=torch.float32, device=device) * std).to(tdtype)
    if peaky_frac > 0.0:
        mask = torch.rand((b,), generator=gen, device=device) < peaky_frac
        k_new[mask] = (k_new[mask].float() * peaky_factor).to(tdtype)
    positions = (seq_lens - 1).clamp(min=0)
    return PagedBatch(name=name, q=q, k_pool=k_pool, v_pool=v_pool,
                      block_table=block_table, seq_lens=seq_lens, k_new=k_new,
                      v_new=v_new, positions=positions,
                      scale=1.0 / math.sqrt(head_dim), block_size=block_size,
                      seed=seed, pages_per_split=pages_per_split,
                      meta={"std": std, "peaky_frac": peaky_frac,
                            "n_peaky": n_peaky, "device": device})


def tiny(device: str = "cpu") -> PagedBatch:
    """1 sequence, 64 tokens, GQA 4, d 64, fp32, 4 pages out of a 16-page pool."""
    return make_batch("tiny", seed=0, dtype="f32", lens=[64], num_q_heads=32,
                      num_kv_heads=8, head_dim=64, block_size=16, num_pages=16,
                      take_pages=4, device=device)


def awkward(device: str = "cpu") -> PagedBatch:
    """Histories {1, 13, 100, 257}, 12 q heads over 4 kv heads, d 48, fp16."""
    return make_batch("awkward", seed=1, dtype="f16", lens=[1, 13, 100, 257],
                      num_q_heads=12, num_kv_heads=4, head_dim=48, block_size=16,
                      num_pages=64, device=device)


LLAMA1B_HISTORIES = (16, 64, 256, 1024, 4096)


def llama1b(history: int, batch: int = 64, device: str = "cpu",
            num_pages: int = 20000) -> PagedBatch:
    """Llama-3.2-1B heads (32 q / 8 kv, d 64), bf16, every sequence at ``history``."""
    return make_batch(f"llama1b_h{history}", seed=2, dtype="bf16",
                      lens=[history] * batch, num_q_heads=32, num_kv_heads=8,
                      head_dim=64, block_size=16, num_pages=num_pages, device=device)


def ragged8b(batch: int = 256, device: str = "cpu", num_pages: int = 160000,
             max_len: int = 8192) -> PagedBatch:
    """Llama-3-8B heads (32 q / 8 kv, d 128), bf16 std 0.5, lengths U[16, max_len]."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(3)
    lens = torch.randint(16, max_len + 1, (batch,), generator=gen).tolist()
    return make_batch("ragged8b", seed=3, dtype="bf16", lens=lens,
                      num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                      num_pages=num_pages, std=0.5, device=device)


LONGCTX_HISTORIES = (32768, 131072)


def longctx(history: int, batch: int = 8, device: str = "cpu") -> PagedBatch:
    """Long histories, d 128, bf16, 1% of keys x8; pool = exactly the pages needed."""
    pages = batch * math.ceil(history / 16)
    return make_batch(f"longctx_h{history}", seed=4, dtype="bf16",
                      lens=[history] * batch, num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=16, num_pages=pages,
                      peaky_frac=0.01, peaky_factor=8.0, pages_per_split=64,
                      device=device)


DENSE_CONTEXTS = (1024, 2048, 4096, 8192, 16384)
DENSE_SPLITS = (1, 8, 16, 32, 64, 128)


def dense(n_ctx: int, batch: int = 4, heads: int = 16, head_dim: int = 64,
          dtype: str = "f16", device: str = "cpu", seed: int = 5) -> PagedBatch:
    """Contiguous K/V: sequence b's pages are b*N/16 .. (b+1)*N/16 - 1, in order."""
    bs = 16
    npg = -(-n_ctx // bs)
    tdtype = DTYPES[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    table = torch.arange(batch * npg, dtype=torch.int32, device=device).reshape(batch, npg)
    q = torch.randn((batch, heads, head_dim), generator=gen, device=device).to(tdtype)
    k_pool = _draw_pool(gen, batch * npg, bs, heads, head_dim, 1.0, tdtype, device)
    v_pool = _draw_pool(gen, batch * npg, bs, heads, head_dim, 1.0, tdtype, device)
    k_new = torch.randn((batch, heads, head_dim), generator=gen, device=device).to(tdtype)
    v_new = torch.randn((batch, heads, head_dim), generator=gen, device=device).to(tdtype)
    seq_lens = torch.full((batch,), n_ctx, dtype=torch.int32, device=device)
    return PagedBatch(name=f"dense_n{n_ctx}", q=q, k_pool=k_pool, v_pool=v_pool,
                      block_table=table, seq_lens=seq_lens, k_new=k_new, v_new=v_new,
                      positions=seq_lens - 1, scale=1.0 / math.sqrt(head_dim), block_size=bs,
                      seed=seed, meta={"dense": True})
