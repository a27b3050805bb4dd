"""pa_decode_splitkv_noalloc: the split-KV read + merge for callers that
cannot allocate device memory.

Such a caller (a plugin whose host framework owns every device allocation,
or a serving loop that may not call cudaMalloc because it can synchronize
the device) cannot hand pa_decode_splitkv the space for its partials.  This
entry point keeps them in a fixed array the library holds in device memory.
These tests call it through the C ABI and check it against the existing
entry points (pa_decode_splitkv followed by pa_merge), on two calls in a
row, so that what one call leaves in the shared array cannot leak into the
next.  The file sorts last so that a run stopping at the first failure has
already run every other test.
"""

import pytest
import torch

import workloads
from helpers import TOL

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _existing(lib, g, pps):
    s = lib.pa_num_splits(g.max_blocks, pps)
    po = torch.empty((g.num_seqs, g.num_q_heads, s, g.head_dim), device=DEV)
    pl = torch.empty((g.num_seqs, g.num_q_heads, s), device=DEV)
    lib.pa_decode_splitkv(po, pl, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens, g.scale,
                          pps)
    out = torch.empty_like(g.q)
    lib.pa_merge(out, po, pl)
    return out


def _noalloc(lib, g, pps):
    out = torch.full_like(g.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    lib.pa_decode_splitkv_noalloc(out, g.q, g.k_pool, g.v_pool, g.block_table, g.seq_lens,
                                  g.scale, pps, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def _close(got, want, dtype):
    tol = TOL[dtype]
    g, w = got.double(), want.double()
    assert torch.isfinite(g).all()
    assert ((g - w).abs() <= tol + tol * w.abs()).all(), float((g - w).abs().max())


CASES = {
    "awkward_f16_pps2": (lambda: workloads.awkward(), 2),
    "llama1b_h1024_pps16": (lambda: workloads.llama1b(1024), 16),
    "longctx_h32768_pps64": (lambda: workloads.longctx(32768, device=DEV), 64),
}


@pytest.mark.parametrize("name", list(CASES))
def test_two_calls_in_a_row_match_the_existing_entry_points(lib, name):
    make, pps = CASES[name]
    g = make().to(DEV)
    want = _existing(lib, g, pps)
    first = _noalloc(lib, g, pps)
    second = _noalloc(lib, g, pps)
    _close(first, want, g.dtype)
    _close(second, want, g.dtype)


def test_a_different_batch_in_between_leaves_no_trace(lib):
    a = workloads.awkward().to(DEV)
    b = workloads.llama1b(256, batch=8).to(DEV)
    want_a = _existing(lib, a, 1)
    want_b = _existing(lib, b, 4)
    _close(_noalloc(lib, a, 1), want_a, a.dtype)
    _close(_noalloc(lib, b, 4), want_b, b.dtype)
    _close(_noalloc(lib, a, 1), want_a, a.dtype)


def test_partials_beyond_the_array_are_refused(lib):
    import paged_kv_cache_184_gb300 as pa
    g = workloads.llama1b(256, batch=64).to(DEV)
    # one page per split: 64 sequences x 32 heads x 16 splits x 65 floats (8.5 MB) fit;
    # 64 x 64 heads x 256 splits x 129 floats (541 MB) do not
    big = workloads.make_batch("big", 5, "bf16", [4096] * 64, 64, 8, 128, 16, 16384, device=DEV)
    with pytest.raises(pa.PaError) as e:
        lib.pa_decode_splitkv_noalloc(torch.empty_like(big.q), big.q, big.k_pool, big.v_pool,
                                      big.block_table, big.seq_lens, big.scale, 1)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    _close(_noalloc(lib, g, 1), _existing(lib, g, 1), g.dtype)


def test_f32_cache_matches_the_existing_entry_points(lib):
    # the fp32 cache runs the CUDA-core read, held to the 1e-5 tolerance
    g = workloads.tiny().to(DEV)
    want = _existing(lib, g, 1)
    _close(_noalloc(lib, g, 1), want, g.dtype)
    _close(_noalloc(lib, g, 1), want, g.dtype)


def test_partials_that_fill_the_array_to_the_byte(lib):
    # 53 sequences x 5 heads x 487 one-page splits: the partial outputs (256 x 129,055 bytes)
    # and the lse (516,220 bytes, rounded up to 516,352) take exactly the array's 32 MiB;
    # one split more is refused before anything is launched
    import paged_kv_cache_184_gb300 as pa
    gen = torch.Generator().manual_seed(13)
    lens = torch.randint(0, 487 * 16 + 1, (53,), generator=gen).tolist()
    lens[0], lens[1] = 487 * 16, 0                 # one full table row, one empty sequence
    pages = sum(-(-n // 16) for n in lens) + 8
    g = workloads.make_batch("exact_fit", 13, "bf16", lens, 5, 1, 64, 16, pages,
                             max_blocks=487).to(DEV)
    want = _existing(lib, g, 1)
    _close(_noalloc(lib, g, 1), want, g.dtype)
    _close(_noalloc(lib, g, 1), want, g.dtype)
    wide = torch.full((53, 488), -1, dtype=torch.int32, device=DEV)
    wide[:, :487] = g.block_table
    with pytest.raises(pa.PaError) as e:
        lib.pa_decode_splitkv_noalloc(torch.empty_like(g.q), g.q, g.k_pool, g.v_pool, wide,
                                      g.seq_lens, g.scale, 1)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_a_second_context_on_the_device_uses_its_own_copy_of_the_array(lib, tmp_path):
    # The array's address belongs to the context the library's module was loaded into.  A
    # child process (no torch) runs the call in the primary context, in a second context it
    # creates on the same device, and in the primary context again; each must match the
    # existing entry points.  (A device reset inside this process is not exercised: torch's
    # allocator would keep pointers into the old context.)
    import os
    import subprocess
    import sys
    import numpy as np

    cases = {"tiny": (workloads.tiny(), 1, 0), "awkward": (workloads.awkward(), 2, 1)}
    arrays, wants = {"cases": np.array(list(cases))}, {}
    for name, (cpu, pps, code) in cases.items():
        for k in ("q", "k_pool", "v_pool", "block_table", "seq_lens"):
            arrays[f"{name}_{k}"] = getattr(cpu, k).numpy()
        arrays[f"{name}_meta"] = np.array([cpu.scale, cpu.block_size, pps, code])
        wants[name] = (_existing(lib, cpu.to(DEV), pps), cpu.dtype)
    inp, outp = tmp_path / "in.npz", tmp_path / "out.npz"
    np.savez(inp, **arrays)
    script = os.path.join(os.path.dirname(os.path.abspath(__file__)), "native",
                          "noalloc_contexts.py")
    r = subprocess.run([sys.executable, script, str(inp), str(outp), lib.LIB_PATH],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    got = np.load(outp)
    for name, (want, dtype) in wants.items():
        for where in ("primary", "second", "primary_again"):
            _close(torch.from_numpy(got[f"{name}_{where}"]).to(DEV), want, dtype)
