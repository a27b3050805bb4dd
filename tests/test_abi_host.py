"""Host-side checks of the C ABI: the library loads, exports what include/pa.h
declares, and rejects bad arguments before launching anything.

No call here reaches a kernel launch: every call is either a pure host
function or one that the validation layer must refuse (or treat as an empty
no-op) before any CUDA call.
"""

import ctypes
import os
import re

import pytest

import paged_kv_cache_184_gb300 as pa

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pa.h")

# non-null, 16-byte aligned stand-ins that are never dereferenced
FAKE = 0x10000
MISALIGNED = 0x10008


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def test_library_builds_and_exports_every_declared_symbol(lib):
    raw = lib.raw()
    names = declared_functions()
    assert set(names) == set(pa.EXPORTED)
    for n in names:
        assert hasattr(raw, n), n


def declared_parameters():
    """{function: [parameter declarations]} from include/pa.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(pa_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", text):
        params = " ".join(params.split())
        out[name] = [] if params in ("", "void") else [x.strip() for x in params.split(",")]
    return out


def _ctype_of(decl):
    if "*" in decl or decl.startswith("pa_stream_t"):
        return ctypes.c_void_p
    for prefix, ct in (("int32_t", ctypes.c_int32), ("float", ctypes.c_float),
                       ("pa_dtype", ctypes.c_int), ("pa_status", ctypes.c_int)):
        if decl.startswith(prefix):
            return ct
    raise AssertionError(f"unmapped parameter type: {decl}")


def test_binding_signatures_match_the_header():
    # the ctypes argument lists have the header's arity and, position by position, its types
    decl = declared_parameters()
    assert set(decl) == set(pa._SIGNATURES)
    for name, (_, args) in pa._SIGNATURES.items():
        assert len(args) == len(decl[name]), name
        for i, (got, d) in enumerate(zip(args, decl[name])):
            assert got == _ctype_of(d), f"{name} argument {i}: {d}"


def test_status_strings_and_version(lib):
    assert lib.pa_status_string(0) == "PA_OK"
    assert lib.pa_status_string(1) == "PA_ERR_INVALID_ARG"
    assert lib.pa_status_string(2) == "PA_ERR_UNSUPPORTED"
    assert lib.pa_status_string(3) == "PA_ERR_CUDA"
    assert lib.pa_status_string(99) == "PA_ERR_UNKNOWN"
    assert "sm_103a" in lib.pa_version()


@pytest.mark.parametrize("mb,pps,want", [(256, 64, 4), (257, 64, 5), (1, 64, 1), (64, 1, 64),
                                          (8192, 64, 128), (0, 64, 0), (5, 0, 0), (-1, 4, 0)])
def test_num_splits(lib, mb, pps, want):
    assert lib.pa_num_splits(mb, pps) == want


def _decode(raw, **kw):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=4, sl=FAKE, b=2, hq=8, hkv=2, d=64,
             bs=16, np_=32, scale=0.125, dt=pa.PA_BF16)
    a.update(kw)
    return raw.pa_decode(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["b"],
                         a["hq"], a["hkv"], a["d"], a["bs"], a["np_"], a["scale"], a["dt"],
                         None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(hq=9, hkv=2), pa.PA_ERR_INVALID_ARG),          # group not integral
    (dict(hkv=0), pa.PA_ERR_INVALID_ARG),
    (dict(d=0), pa.PA_ERR_INVALID_ARG),
    (dict(d=36), pa.PA_ERR_UNSUPPORTED),                 # 72 bytes: not a multiple of 16
    (dict(d=512), pa.PA_ERR_UNSUPPORTED),                # beyond 256
    (dict(d=6, dt=pa.PA_F32), pa.PA_ERR_UNSUPPORTED),    # 24 bytes
    (dict(hq=18, hkv=1), pa.PA_ERR_UNSUPPORTED),         # group of 18
    (dict(hq=12, hkv=1, dt=pa.PA_F32), pa.PA_ERR_UNSUPPORTED),   # group 12 needs f16/bf16
    (dict(hq=12, hkv=1, d=80), pa.PA_ERR_UNSUPPORTED),   # ... and a tensor-core head_dim
    (dict(hq=16, hkv=1, b=0), pa.PA_OK),                 # group 16, bf16, d 64
    (dict(bs=12), pa.PA_ERR_INVALID_ARG),                # not a power of two
    (dict(bs=0), pa.PA_ERR_INVALID_ARG),
    (dict(bs=2048), pa.PA_ERR_UNSUPPORTED),
    (dict(mb=0), pa.PA_ERR_INVALID_ARG),
    (dict(np_=0), pa.PA_ERR_INVALID_ARG),
    (dict(b=-1), pa.PA_ERR_INVALID_ARG),
    (dict(b=70000), pa.PA_ERR_UNSUPPORTED),
    (dict(dt=7), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pa.PA_ERR_INVALID_ARG),
    (dict(q=None), pa.PA_ERR_INVALID_ARG),
    (dict(sl=None), pa.PA_ERR_INVALID_ARG),
    (dict(k=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(out=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),                               # empty batch: nothing to launch
])
def test_decode_validation(lib, kw, want):
    assert _decode(lib.raw(), **kw) == want


def _split(raw, **kw):
    a = dict(po=FAKE, pl=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=10, sl=FAKE, b=2, hq=8, hkv=2,
             d=64, bs=16, np_=32, scale=0.125, pps=4, ms=3, dt=pa.PA_F16)
    a.update(kw)
    return raw.pa_decode_splitkv(a["po"], a["pl"], a["q"], a["k"], a["v"], a["bt"], a["mb"],
                                 a["sl"], a["b"], a["hq"], a["hkv"], a["d"], a["bs"], a["np_"],
                                 a["scale"], a["pps"], a["ms"], a["dt"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(ms=2), pa.PA_ERR_INVALID_ARG),                 # 10 pages / 4 per split needs 3
    (dict(pps=0), pa.PA_ERR_INVALID_ARG),
    (dict(pl=None), pa.PA_ERR_INVALID_ARG),
    (dict(po=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(hq=6, hkv=4), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),
])
def test_splitkv_validation(lib, kw, want):
    assert _split(lib.raw(), **kw) == want


@pytest.mark.parametrize("args,want", [
    ((FAKE, FAKE, FAKE, 2, 4, 0, 64, pa.PA_BF16), pa.PA_ERR_INVALID_ARG),   # no splits
    ((FAKE, FAKE, FAKE, 2, 4, 3, 0, pa.PA_BF16), pa.PA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 2, 4, 3, 320, pa.PA_BF16), pa.PA_ERR_UNSUPPORTED),
    ((FAKE, FAKE, FAKE, 2, 4, 3, 64, 5), pa.PA_ERR_INVALID_ARG),
    ((None, FAKE, FAKE, 2, 4, 3, 64, pa.PA_BF16), pa.PA_ERR_INVALID_ARG),
    ((FAKE, FAKE, FAKE, 0, 4, 3, 64, pa.PA_BF16), pa.PA_OK),
    ((FAKE, FAKE, FAKE, 2, 4, 3, 6, pa.PA_F32), pa.PA_ERR_UNSUPPORTED),    # not float4 rows
    ((FAKE, MISALIGNED, FAKE, 2, 4, 3, 64, pa.PA_BF16), pa.PA_ERR_INVALID_ARG),
])
def test_merge_validation(lib, args, want):
    assert lib.raw().pa_merge(*args, None) == want


def _append(raw, **kw):
    a = dict(kn=FAKE, vn=FAKE, kp=FAKE, vp=FAKE, bt=FAKE, ns=4, mb=8, sid=None, pos=FAKE, nt=4,
             np_=32, hkv=8, d=64, bs=16, dt=pa.PA_BF16)
    a.update(kw)
    return raw.pa_cache_append(a["kn"], a["vn"], a["kp"], a["vp"], a["bt"], a["ns"], a["mb"],
                               a["sid"], a["pos"], a["nt"], a["np_"], a["hkv"], a["d"], a["bs"],
                               a["dt"], None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(nt=5), pa.PA_ERR_INVALID_ARG),                 # token i -> seq i needs nt <= ns
    (dict(bs=3), pa.PA_ERR_INVALID_ARG),
    (dict(bs=4096), pa.PA_ERR_UNSUPPORTED),
    (dict(hkv=1, d=4), pa.PA_ERR_UNSUPPORTED),           # 8-byte rows
    (dict(pos=None), pa.PA_ERR_INVALID_ARG),
    (dict(kp=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(nt=-1), pa.PA_ERR_INVALID_ARG),
    (dict(dt=9), pa.PA_ERR_INVALID_ARG),
    (dict(nt=0), pa.PA_OK),
    (dict(nt=0, kn=None), pa.PA_OK),                     # empty append touches nothing
])
def test_append_validation(lib, kw, want):
    assert _append(lib.raw(), **kw) == want


def test_binding_rejects_host_tensors(lib):
    import torch
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    kp = torch.zeros(2, 16, 1, 64, dtype=torch.bfloat16)
    bt = torch.zeros(1, 2, dtype=torch.int32)
    sl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        lib.pa_decode(torch.empty_like(q), q, kp, kp, bt, sl, 0.125)


def test_missing_library_raises_with_no_fallback(lib, monkeypatch, tmp_path):
    # the binding has no other implementation: without libpa.so every entry point fails
    monkeypatch.setattr(pa, "_lib", None)
    monkeypatch.setattr(pa, "LIB_PATH", str(tmp_path / "libpa.so"))
    with pytest.raises(RuntimeError, match="not built"):
        pa.load(build=False)
    with pytest.raises(RuntimeError, match="not built"):
        pa.pa_num_splits(10, 2)


def test_binding_raises_on_bad_status(lib):
    assert isinstance(pa.PaError("pa_decode", 2), RuntimeError)
    assert "PA_ERR_UNSUPPORTED" in str(pa.PaError("pa_decode", 2))


# 53 sequences x 5 heads x 487 splits = 129,055 partial rows: 256 x 129,055 bytes of outputs
# and 516,220 of lse rounded up to 516,352 fill the 32 MiB array exactly; 488 splits do not
EXACT_FIT = dict(b=53, hq=5, hkv=1, d=64, mb=487, pps=1)


def test_exact_fit_shape_fills_the_array():
    rows = 53 * 5 * 487
    align = lambda x: (x + 255) // 256 * 256
    assert align(rows * 64 * 4) + align(rows * 4) == pa.PA_NOALLOC_SCRATCH_BYTES
    rows += 53 * 5
    assert align(rows * 64 * 4) + align(rows * 4) > pa.PA_NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("kw,want", [
    (dict(pps=0), pa.PA_ERR_INVALID_ARG),
    (dict(b=-1), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),
    # 64 x 32 x 8192 splits x 65 floats: far beyond the fixed partials array
    (dict(b=64, mb=8192, pps=1), pa.PA_ERR_UNSUPPORTED),
    # the read's own checks come first, as in pa_decode_splitkv: an empty batch with a bad
    # shape, and an oversized batch with a bad group, are both invalid arguments
    (dict(b=0, hkv=0), pa.PA_ERR_INVALID_ARG),
    (dict(b=0, bs=24), pa.PA_ERR_INVALID_ARG),
    (dict(b=0, dt=9), pa.PA_ERR_INVALID_ARG),
    (dict(b=64, mb=8192, pps=1, hq=9, hkv=2), pa.PA_ERR_INVALID_ARG),
    (dict(b=0, d=512), pa.PA_ERR_UNSUPPORTED),
    (dict(EXACT_FIT, mb=488), pa.PA_ERR_UNSUPPORTED),    # one split past the exact fit
    (dict(out=None), pa.PA_ERR_INVALID_ARG),             # refused before anything launches
    (dict(out=MISALIGNED), pa.PA_ERR_INVALID_ARG),
])
def test_noalloc_validation_before_any_device_call(lib, kw, want):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=10, sl=FAKE, b=2, hq=32, hkv=8, d=64,
             bs=16, np_=32, scale=0.125, pps=4, dt=pa.PA_BF16)
    a.update(kw)
    st = lib.raw().pa_decode_splitkv_noalloc(
        a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["b"], a["hq"], a["hkv"],
        a["d"], a["bs"], a["np_"], a["scale"], a["pps"], a["dt"], None, None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(nq=0), pa.PA_ERR_INVALID_ARG),
    (dict(dt=pa.PA_F32), pa.PA_ERR_UNSUPPORTED),          # tensor-core read only
    (dict(d=256), pa.PA_ERR_UNSUPPORTED),
    (dict(d=80), pa.PA_ERR_UNSUPPORTED),
    (dict(hq=9, hkv=2), pa.PA_ERR_INVALID_ARG),
    (dict(q=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),
    (dict(b=0, hq=16, hkv=1, nq=4096), pa.PA_OK),
    # (query, head) rows per kv head past 2^30 are refused before any 32-bit product
    (dict(nq=(1 << 28) + 1), pa.PA_ERR_UNSUPPORTED),
    (dict(nq=2**31 - 1, hq=16, hkv=1), pa.PA_ERR_UNSUPPORTED),
])
def test_chunk_validation(lib, kw, want):
    a = dict(out=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=4, sl=FAKE, b=2, nq=8, hq=8, hkv=2,
             d=64, bs=16, np_=32, scale=0.125, dt=pa.PA_BF16)
    a.update(kw)
    st = lib.raw().pa_decode_chunk(a["out"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"],
                                   a["b"], a["nq"], a["hq"], a["hkv"], a["d"], a["bs"], a["np_"],
                                   a["scale"], a["dt"], None, None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(dt=pa.PA_F32), pa.PA_ERR_UNSUPPORTED),          # tensor-core read only
    (dict(slots=0), pa.PA_ERR_INVALID_ARG),
    (dict(slots=40000), pa.PA_ERR_INVALID_ARG),
    (dict(n=0), pa.PA_ERR_INVALID_ARG),                   # every sequence needs an item
    (dict(items=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),
])
def test_work_validation(lib, kw, want):
    a = dict(po=FAKE, pl=FAKE, items=FAKE, n=10, slots=4, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=4,
             sl=FAKE, b=2, hq=8, hkv=2, d=64, bs=16, np_=32, scale=0.125, dt=pa.PA_BF16)
    a.update(kw)
    st = lib.raw().pa_decode_work(a["po"], a["pl"], a["items"], a["n"], a["slots"], a["q"],
                                  a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["b"], a["hq"],
                                  a["hkv"], a["d"], a["bs"], a["np_"], a["scale"], a["dt"],
                                  None, None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(nq=0), pa.PA_ERR_INVALID_ARG),
    (dict(pps=0), pa.PA_ERR_INVALID_ARG),
    (dict(dt=pa.PA_F32), pa.PA_ERR_UNSUPPORTED),          # tensor-core read only
    (dict(d=80), pa.PA_ERR_UNSUPPORTED),
    (dict(ms=3), pa.PA_ERR_INVALID_ARG),                  # 4 pages, 1 per split: 4 needed
    (dict(ms=70000), pa.PA_ERR_UNSUPPORTED),              # the split is the grid's z index
    (dict(po=MISALIGNED), pa.PA_ERR_INVALID_ARG),
    (dict(pl=None), pa.PA_ERR_INVALID_ARG),
    (dict(b=0), pa.PA_OK),
    (dict(nq=2**31 - 1, hq=16, hkv=1), pa.PA_ERR_UNSUPPORTED),
])
def test_chunk_splitkv_validation(lib, kw, want):
    a = dict(po=FAKE, pl=FAKE, q=FAKE, k=FAKE, v=FAKE, bt=FAKE, mb=4, sl=FAKE, b=2, nq=8, hq=8,
             hkv=2, d=64, bs=16, np_=32, scale=0.125, pps=1, ms=4, dt=pa.PA_BF16)
    a.update(kw)
    st = lib.raw().pa_decode_chunk_splitkv(
        a["po"], a["pl"], a["q"], a["k"], a["v"], a["bt"], a["mb"], a["sl"], a["b"], a["nq"],
        a["hq"], a["hkv"], a["d"], a["bs"], a["np_"], a["scale"], a["pps"], a["ms"], a["dt"],
        None, None)
    assert st == want


def test_binding_merge_and_chunk_split_shape_checks(lib):
    # shape checks of the binding raise before any pointer is taken or any call is made
    import torch
    po = torch.zeros(2, 3, 4, 5, 64)              # [B, n_q, Hq, S, d]
    pl = torch.zeros(2, 3, 4, 5)
    with pytest.raises(ValueError):                # out must be [B, n_q, Hq, d]
        lib.pa_merge(torch.zeros(2, 3, 4, 32, dtype=torch.bfloat16), po, pl)
    with pytest.raises(ValueError):                # lse must match the leading axes
        lib.pa_merge(torch.zeros(2, 3, 4, 64, dtype=torch.bfloat16), po, torch.zeros(2, 3, 5, 5))
    with pytest.raises(ValueError):                # partials need at least [B, Hq, S, d]
        lib.pa_merge(torch.zeros(4, 64), torch.zeros(4, 5, 64), torch.zeros(4, 5))
    q = torch.zeros(2, 3, 4, 64, dtype=torch.bfloat16)
    kp = torch.zeros(8, 16, 1, 64, dtype=torch.bfloat16)
    bt = torch.zeros(2, 4, dtype=torch.int32)
    sl = torch.ones(2, dtype=torch.int32)
    with pytest.raises(ValueError):                # partials [B, n_q, Hq, S, d] with S = lse's
        lib.pa_decode_chunk_splitkv(torch.zeros(2, 3, 4, 6, 64), pl, q, kp, kp, bt, sl, 0.125, 1)
    with pytest.raises(ValueError):                # head_dim of q and the pools must agree
        lib.pa_decode_chunk_splitkv(po, pl, torch.zeros(2, 3, 4, 32, dtype=torch.bfloat16), kp,
                                    kp, bt, sl, 0.125, 1)


# ---- the binding checks every row count the C ABI cannot see -------------------------


def _cpu_batch(b=2, hq=8, hkv=2, d=64, mb=4, nq=None):
    import torch
    q = torch.zeros((b, hq, d) if nq is None else (b, nq, hq, d), dtype=torch.bfloat16)
    kp = torch.zeros(16, 16, hkv, d, dtype=torch.bfloat16)
    bt = torch.zeros(b, mb, dtype=torch.int32)
    sl = torch.ones(b, dtype=torch.int32)
    return q, kp, bt, sl


@pytest.mark.parametrize("what", ["short_table", "long_table", "short_lens", "long_lens",
                                  "flat_table"])
def test_binding_checks_table_and_lens_rows_of_every_read(lib, what):
    import torch

    def bad(bt, sl):
        if what == "short_table":
            return bt[:1], sl, "block_table"
        if what == "long_table":
            return torch.zeros(3, 4, dtype=torch.int32), sl, "block_table"
        if what == "short_lens":
            return bt, sl[:1], "seq_lens"
        if what == "long_lens":
            return bt, torch.ones(3, dtype=torch.int32), "seq_lens"
        return bt.reshape(-1), sl, "block_table"

    q, kp, bt, sl = _cpu_batch()
    bt, sl, name = bad(bt, sl)
    po, pl = torch.zeros(2, 8, 4, 64), torch.zeros(2, 8, 4)
    calls = {
        "pa_decode": lambda: lib.pa_decode(torch.empty_like(q), q, kp, kp, bt, sl, 0.125),
        "pa_decode_splitkv": lambda: lib.pa_decode_splitkv(po, pl, q, kp, kp, bt, sl, 0.125, 1),
        "pa_decode_splitkv_noalloc": lambda: lib.pa_decode_splitkv_noalloc(
            torch.empty_like(q), q, kp, kp, bt, sl, 0.125, 1),
        "pa_decode_work": lambda: lib.pa_decode_work(
            po, pl, torch.zeros(2, 4, dtype=torch.int32), q, kp, kp, bt, sl, 0.125),
    }
    qc, _, _, _ = _cpu_batch(nq=3)
    poc, plc = torch.zeros(2, 3, 8, 4, 64), torch.zeros(2, 3, 8, 4)
    calls["pa_decode_chunk"] = lambda: lib.pa_decode_chunk(torch.empty_like(qc), qc, kp, kp, bt,
                                                           sl, 0.125)
    calls["pa_decode_chunk_splitkv"] = lambda: lib.pa_decode_chunk_splitkv(
        poc, plc, qc, kp, kp, bt, sl, 0.125, 1)
    for fn, call in calls.items():
        with pytest.raises(ValueError, match=f"{fn}: {name} must be"):
            call()


def test_binding_checks_append_rows(lib):
    import torch
    kp = torch.zeros(16, 16, 2, 64, dtype=torch.bfloat16)
    kn = torch.zeros(3, 2, 64, dtype=torch.bfloat16)
    bt = torch.zeros(3, 4, dtype=torch.int32)
    pos = torch.zeros(3, dtype=torch.int32)
    with pytest.raises(ValueError, match="positions must be"):
        lib.pa_cache_append(kn, kn, kp, kp, bt, pos[:2])
    with pytest.raises(ValueError, match="seq_ids must be"):
        lib.pa_cache_append(kn, kn, kp, kp, bt, pos, seq_ids=torch.zeros(4, dtype=torch.int32))
    with pytest.raises(ValueError, match="a row per token"):
        lib.pa_cache_append(kn, kn, kp, kp, bt[:2], pos)
    with pytest.raises(ValueError, match="block_table must be"):
        lib.pa_cache_append(kn, kn, kp, kp, bt.reshape(-1), pos)


@pytest.mark.parametrize("items,match", [
    ([[2, 0, 16, 1 << 16], [0, 0, 16, 1 << 16]], "outside"),           # sequence 2 of 2
    ([[-1, 0, 16, 1 << 16], [1, 0, 16, 1 << 16]], "outside"),
    ([[0, 0, 16, (5 << 16) | 4], [1, 0, 16, 1 << 16]], "max_slots"),   # 5 slots of 4
    ([[0, 0, 16, (1 << 16) | 1], [1, 0, 16, 1 << 16]], "max_slots"),   # slot 1 of 1
])
def test_binding_checks_work_items_on_their_host_copy(lib, items, match):
    import torch
    q, kp, bt, sl = _cpu_batch()
    po, pl = torch.zeros(2, 8, 4, 64), torch.zeros(2, 8, 4)
    host = torch.tensor(items, dtype=torch.int32)
    with pytest.raises(ValueError, match=match):
        lib.pa_decode_work(po, pl, host.clone(), q, kp, kp, bt, sl, 0.125, items_host=host)
