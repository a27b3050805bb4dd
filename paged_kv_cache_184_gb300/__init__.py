"""Python binding of libpa.so, the GB300 paged KV-cache decode-attention library.

Argument marshalling only: every function here takes torch tensors, checks
that they are contiguous device tensors, reads their shapes, and passes raw
pointers and sizes to the C ABI declared in include/pa.h, on the current
CUDA stream.  All arithmetic runs in the library's CUDA kernels; there is
no other implementation to fall back on, so a missing library raises.

The names match the C ABI: pa_cache_append, pa_decode, pa_decode_splitkv,
pa_merge, pa_decode_chunk, pa_decode_chunk_splitkv, pa_plan_work, pa_decode_work,
pa_decode_splitkv_noalloc, pa_num_splits, pa_status_string, pa_version, and the
test hook pa_test_set_withhold_tiles.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

LIB_PATH = _build.LIB_PATH

PA_OK, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_CUDA = 0, 1, 2, 3
PA_F32, PA_F16, PA_BF16 = 0, 1, 2
PA_DEV_OK, PA_DEV_BAD_PAGE, PA_DEV_BAD_POSITION, PA_DEV_BAD_SEQ_LEN, PA_DEV_BAD_SEQ_ID = 0, 1, 2, 3, 4
PA_DEV_BAD_ITEM, PA_DEV_TIMEOUT = 5, 6

EXPORTED = ("pa_status_string", "pa_version", "pa_num_splits", "pa_cache_append",
            "pa_decode", "pa_decode_splitkv", "pa_merge", "pa_decode_splitkv_noalloc",
            "pa_decode_chunk", "pa_decode_chunk_splitkv", "pa_plan_work", "pa_decode_work",
            "pa_test_set_withhold_tiles")

# bytes of the library-owned partials array behind pa_decode_splitkv_noalloc
PA_NOALLOC_SCRATCH_BYTES = 32 << 20

_lib: Optional[ctypes.CDLL] = None

_p = ctypes.c_void_p
_i = ctypes.c_int32
_f = ctypes.c_float

_SIGNATURES = {
    "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pa_version": (ctypes.c_char_p, []),
    "pa_num_splits": (_i, [_i, _i]),
    "pa_cache_append": (ctypes.c_int, [_p, _p, _p, _p, _p, _i, _i, _p, _p, _i, _i, _i, _i, _i,
                                       ctypes.c_int, _p, _p]),
    "pa_decode": (ctypes.c_int, [_p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _f,
                                 ctypes.c_int, _p, _p]),
    "pa_decode_splitkv": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i,
                                         _f, _i, _i, ctypes.c_int, _p, _p]),
    "pa_merge": (ctypes.c_int, [_p, _p, _p, _i, _i, _i, _i, ctypes.c_int, _p]),
    "pa_plan_work": (_i, [_p, _i, _i, _i, _i, _i, _p, _i, _p]),
    "pa_decode_work": (ctypes.c_int, [_p, _p, _p, _i, _i, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i,
                                      _i, _f, ctypes.c_int, _p, _p]),
    "pa_decode_chunk": (ctypes.c_int, [_p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _i, _i, _f,
                                       ctypes.c_int, _p, _p]),
    "pa_decode_chunk_splitkv": (ctypes.c_int, [_p, _p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i,
                                               _i, _i, _f, _i, _i, ctypes.c_int, _p, _p]),
    "pa_decode_splitkv_noalloc": (ctypes.c_int, [_p, _p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i,
                                                 _i, _f, _i, ctypes.c_int, _p, _p]),
    "pa_test_set_withhold_tiles": (None, [_i]),
}


class PaError(RuntimeError):
    """A C-ABI call returned a status other than PA_OK."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status} ({pa_status_string(status)})")


def load(build: bool = True) -> ctypes.CDLL:
    """Load libpa.so (building it first when asked and out of date)."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libpa.so not built at {LIB_PATH}; run paged_kv_cache_184_gb300._build")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def raw() -> ctypes.CDLL:
    """The loaded ctypes library, for callers that pass raw pointers."""
    return load()


def _dtype_code(t) -> int:
    import torch
    codes = {torch.float32: PA_F32, torch.float16: PA_F16, torch.bfloat16: PA_BF16}
    if t.dtype not in codes:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return codes[t.dtype]


def _ptr(t, name: str, dtype=None, allow_none: bool = False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check_batch(fn: str, b: int, block_table, seq_lens) -> None:
    """The table and the lengths must have exactly one row per sequence of the batch:
    the C ABI carries no row count for them, so a short tensor would be read past
    its end."""
    if block_table.dim() != 2 or block_table.shape[0] != b:
        raise ValueError(f"{fn}: block_table must be [{b}, max_blocks], got "
                         f"{list(block_table.shape)}")
    if seq_lens.dim() != 1 or seq_lens.shape[0] != b:
        raise ValueError(f"{fn}: seq_lens must be [{b}], got {list(seq_lens.shape)}")


def _check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PaError(fn, status)


def pa_status_string(status: int) -> str:
    return load().pa_status_string(status).decode()


def pa_version() -> str:
    return load().pa_version().decode()


def pa_num_splits(max_blocks_per_seq: int, pages_per_split: int) -> int:
    return int(load().pa_num_splits(max_blocks_per_seq, pages_per_split))


def pa_test_set_withhold_tiles(on: bool) -> None:
    """Test hook: while on, the warp-specialized chunk read loads no key tile and its
    bounded waits run out (PA_DEV_TIMEOUT, zeroed outputs)."""
    load().pa_test_set_withhold_tiles(1 if on else 0)


def pa_cache_append(k_new, v_new, k_pool, v_pool, block_table, positions, seq_ids=None,
                    dev_err=None, stream=None) -> None:
    """Scatter k_new/v_new [T, Hkv, d] into their page slots of k_pool/v_pool."""
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape or k_new.shape[1:] != (hkv, d):
        raise ValueError("pa_cache_append: inconsistent K/V shapes")
    t = k_new.shape[0]
    if block_table.dim() != 2:
        raise ValueError("pa_cache_append: block_table must be [num_seqs, max_blocks]")
    if positions.dim() != 1 or positions.shape[0] != t:
        raise ValueError(f"pa_cache_append: positions must be [{t}], got {list(positions.shape)}")
    if seq_ids is not None and (seq_ids.dim() != 1 or seq_ids.shape[0] != t):
        raise ValueError(f"pa_cache_append: seq_ids must be [{t}], got {list(seq_ids.shape)}")
    if seq_ids is None and t > block_table.shape[0]:
        raise ValueError("pa_cache_append: without seq_ids token i belongs to sequence i, so "
                         "the table needs a row per token")
    dt = k_pool.dtype
    st = lib.pa_cache_append(
        _ptr(k_new, "k_new", dt), _ptr(v_new, "v_new", dt), _ptr(k_pool, "k_pool", dt),
        _ptr(v_pool, "v_pool", dt), _ptr(block_table, "block_table", torch.int32),
        block_table.shape[0], block_table.shape[1],
        _ptr(seq_ids, "seq_ids", torch.int32, allow_none=True),
        _ptr(positions, "positions", torch.int32), k_new.shape[0], num_pages, hkv, d,
        block_size, _dtype_code(k_pool), _ptr(dev_err, "dev_err", torch.int32, allow_none=True),
        _stream(stream))
    _check("pa_cache_append", st)


def pa_decode(out, q, k_pool, v_pool, block_table, seq_lens, scale: float, dev_err=None,
              stream=None) -> None:
    """out[b, h] = softmax(scale * q[b, h] . K_b) V_b over the paged history."""
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, hq, dq = q.shape
    if dq != d or out.shape != q.shape or v_pool.shape != k_pool.shape:
        raise ValueError("pa_decode: inconsistent shapes")
    _check_batch("pa_decode", b, block_table, seq_lens)
    dt = q.dtype
    st = lib.pa_decode(
        _ptr(out, "out", dt), _ptr(q, "q", dt), _ptr(k_pool, "k_pool", dt),
        _ptr(v_pool, "v_pool", dt), _ptr(block_table, "block_table", torch.int32),
        block_table.shape[1], _ptr(seq_lens, "seq_lens", torch.int32), b, hq, hkv, d,
        block_size, num_pages, float(scale), _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode", st)


def pa_decode_splitkv(partial_out, partial_lse, q, k_pool, v_pool, block_table, seq_lens,
                      scale: float, pages_per_split: int, dev_err=None, stream=None) -> None:
    """Per-split partial outputs [B, Hq, S, d] and lse [B, Hq, S] (float32)."""
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, hq, _ = q.shape
    max_splits = partial_lse.shape[2]
    if partial_out.shape != (b, hq, max_splits, d) or partial_lse.shape != (b, hq, max_splits):
        raise ValueError("pa_decode_splitkv: partial shapes must be [B,Hq,S,d] and [B,Hq,S]")
    if v_pool.shape != k_pool.shape:
        raise ValueError("pa_decode_splitkv: inconsistent shapes")
    _check_batch("pa_decode_splitkv", b, block_table, seq_lens)
    dt = q.dtype
    st = lib.pa_decode_splitkv(
        _ptr(partial_out, "partial_out", torch.float32),
        _ptr(partial_lse, "partial_lse", torch.float32), _ptr(q, "q", dt),
        _ptr(k_pool, "k_pool", dt), _ptr(v_pool, "v_pool", dt),
        _ptr(block_table, "block_table", torch.int32), block_table.shape[1],
        _ptr(seq_lens, "seq_lens", torch.int32), b, hq, hkv, d, block_size, num_pages,
        float(scale), int(pages_per_split), max_splits, _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode_splitkv", st)


def pa_decode_chunk(out, q, k_pool, v_pool, block_table, seq_lens, scale: float, dev_err=None,
                    stream=None) -> None:
    """Causal read of q [B, n_q, Hq, d]: query i sees tokens 0 .. seq_len - n_q + i."""
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, nq, hq, dq = q.shape
    if dq != d or out.shape != q.shape or v_pool.shape != k_pool.shape:
        raise ValueError("pa_decode_chunk: inconsistent shapes")
    _check_batch("pa_decode_chunk", b, block_table, seq_lens)
    dt = q.dtype
    st = lib.pa_decode_chunk(
        _ptr(out, "out", dt), _ptr(q, "q", dt), _ptr(k_pool, "k_pool", dt),
        _ptr(v_pool, "v_pool", dt), _ptr(block_table, "block_table", torch.int32),
        block_table.shape[1], _ptr(seq_lens, "seq_lens", torch.int32), b, nq, hq, hkv, d,
        block_size, num_pages, float(scale), _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode_chunk", st)


def pa_decode_chunk_splitkv(partial_out, partial_lse, q, k_pool, v_pool, block_table, seq_lens,
                            scale: float, pages_per_split: int, dev_err=None,
                            stream=None) -> None:
    """Per-split partials of the chunked read: [B, n_q, Hq, S, d] and [B, n_q, Hq, S] (float32).

    pa_merge(out, partial_out, partial_lse) then gives pa_decode_chunk's out.
    """
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, nq, hq, dq = q.shape
    max_splits = partial_lse.shape[-1]
    if (dq != d or v_pool.shape != k_pool.shape or
            partial_out.shape != (b, nq, hq, max_splits, d) or
            partial_lse.shape != (b, nq, hq, max_splits)):
        raise ValueError("pa_decode_chunk_splitkv: partial shapes must be [B,n_q,Hq,S,d] and "
                         "[B,n_q,Hq,S]")
    _check_batch("pa_decode_chunk_splitkv", b, block_table, seq_lens)
    dt = q.dtype
    st = lib.pa_decode_chunk_splitkv(
        _ptr(partial_out, "partial_out", torch.float32),
        _ptr(partial_lse, "partial_lse", torch.float32), _ptr(q, "q", dt),
        _ptr(k_pool, "k_pool", dt), _ptr(v_pool, "v_pool", dt),
        _ptr(block_table, "block_table", torch.int32), block_table.shape[1],
        _ptr(seq_lens, "seq_lens", torch.int32), b, nq, hq, hkv, d, block_size, num_pages,
        float(scale), int(pages_per_split), max_splits, _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode_chunk_splitkv", st)


def pa_plan_work(seq_lens, num_kv_heads: int, block_size: int, target_ctas: int,
                 min_pages_per_item: int = 16):
    """Host work plan of a ragged batch: (items int32 [n, 4] on the CPU, max_slots).

    seq_lens is the host copy of the lengths (a CPU tensor or a sequence).
    """
    import torch
    lib = load()
    lens = torch.as_tensor(seq_lens, dtype=torch.int32).contiguous()
    if lens.is_cuda:
        raise ValueError("pa_plan_work plans from the host copy of the lengths")
    pages = int(((lens.to(torch.int64) + block_size - 1) // block_size).sum())
    cap = lens.numel() + pages // max(1, min_pages_per_item) + 1
    items = torch.empty((cap, 4), dtype=torch.int32)
    slots = ctypes.c_int32(0)
    n = lib.pa_plan_work(lens.data_ptr(), lens.numel(), num_kv_heads, block_size, target_ctas,
                         min_pages_per_item, items.data_ptr(), cap, ctypes.byref(slots))
    if n < 0:
        raise PaError("pa_plan_work", PA_ERR_INVALID_ARG)
    return items[:n].clone(), int(slots.value)


def pa_decode_work(partial_out, partial_lse, items, q, k_pool, v_pool, block_table, seq_lens,
                   scale: float, dev_err=None, stream=None, items_host=None) -> None:
    """Split read over a planned work list (items: device int32 [n, 4] from pa_plan_work).

    items_host, the plan's host copy when the caller still has it, is checked
    against the batch before the launch: same shape, sequence ids in [0, B) and
    slots below max_slots.
    """
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, hq, _ = q.shape
    max_slots = partial_lse.shape[2]
    if partial_out.shape != (b, hq, max_slots, d) or partial_lse.shape != (b, hq, max_slots):
        raise ValueError("pa_decode_work: partial shapes must be [B,Hq,S,d] and [B,Hq,S]")
    if items.dim() != 2 or items.shape[1] != 4:
        raise ValueError("pa_decode_work: items must be [n, 4]")
    if v_pool.shape != k_pool.shape:
        raise ValueError("pa_decode_work: inconsistent shapes")
    _check_batch("pa_decode_work", b, block_table, seq_lens)
    if items_host is not None:
        h = torch.as_tensor(items_host)
        if tuple(h.shape) != tuple(items.shape):
            raise ValueError("pa_decode_work: items_host and items differ in shape")
        if h.numel():
            seq, slot, count = h[:, 0], h[:, 3] & 0xFFFF, h[:, 3] >> 16
            if bool(((seq < 0) | (seq >= b)).any()):
                raise ValueError(f"pa_decode_work: an item names a sequence outside [0, {b})")
            if bool(((slot >= count) | (count > max_slots)).any()):
                raise ValueError("pa_decode_work: an item's slot or count exceeds max_slots")
    dt = q.dtype
    st = lib.pa_decode_work(
        _ptr(partial_out, "partial_out", torch.float32),
        _ptr(partial_lse, "partial_lse", torch.float32), _ptr(items, "items", torch.int32),
        items.shape[0], max_slots, _ptr(q, "q", dt), _ptr(k_pool, "k_pool", dt),
        _ptr(v_pool, "v_pool", dt), _ptr(block_table, "block_table", torch.int32),
        block_table.shape[1], _ptr(seq_lens, "seq_lens", torch.int32), b, hq, hkv, d, block_size,
        num_pages, float(scale), _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode_work", st)


def pa_merge(out, partial_out, partial_lse, stream=None) -> None:
    """out[..., h] = sum_s w_s partial_out[..., h, s] / sum_s w_s, w_s = exp(lse_s - max lse).

    partial_out [..., Hq, S, d], partial_lse [..., Hq, S], out [..., Hq, d]: the
    leading axes ([B] for decode, [B, n_q] for a chunk) are one row axis.
    """
    import torch
    lib = load()
    if partial_out.dim() < 4:
        raise ValueError("pa_merge: partial_out must be [..., Hq, S, d]")
    *lead, hq, s, d = partial_out.shape
    if (tuple(out.shape) != (*lead, hq, d) or tuple(partial_lse.shape) != (*lead, hq, s)):
        raise ValueError("pa_merge: inconsistent shapes")
    b = 1
    for x in lead:
        b *= x
    st = lib.pa_merge(_ptr(out, "out"), _ptr(partial_out, "partial_out", torch.float32),
                      _ptr(partial_lse, "partial_lse", torch.float32), b, hq, s, d,
                      _dtype_code(out), _stream(stream))
    _check("pa_merge", st)


def pa_decode_splitkv_noalloc(out, q, k_pool, v_pool, block_table, seq_lens, scale: float,
                              pages_per_split: int, dev_err=None, stream=None) -> None:
    """Split-KV read + merge into ``out`` with no scratch from the caller.

    For callers that cannot allocate device memory (a plugin inside a
    framework that owns all allocations, a serving loop that must not call
    cudaMalloc).  The partials live in a fixed library-owned device array of
    PA_NOALLOC_SCRATCH_BYTES; a batch whose partials do not fit raises
    PaError with PA_ERR_UNSUPPORTED.  All calls on a device share that array,
    so calls that overlap on the GPU race.
    """
    import torch
    lib = load()
    num_pages, block_size, hkv, d = k_pool.shape
    b, hq, dq = q.shape
    if dq != d or out.shape != q.shape or v_pool.shape != k_pool.shape:
        raise ValueError("pa_decode_splitkv_noalloc: inconsistent shapes")
    _check_batch("pa_decode_splitkv_noalloc", b, block_table, seq_lens)
    dt = q.dtype
    st = lib.pa_decode_splitkv_noalloc(
        _ptr(out, "out", dt), _ptr(q, "q", dt), _ptr(k_pool, "k_pool", dt),
        _ptr(v_pool, "v_pool", dt), _ptr(block_table, "block_table", torch.int32),
        block_table.shape[1], _ptr(seq_lens, "seq_lens", torch.int32), b, hq, hkv, d,
        block_size, num_pages, float(scale), int(pages_per_split), _dtype_code(q),
        _ptr(dev_err, "dev_err", torch.int32, allow_none=True), _stream(stream))
    _check("pa_decode_splitkv_noalloc", st)
