"""Host cost of a launch through the C ABI.

A serving step issues a few short reads (8-12 us of device time at short
histories), so the host work per call matters.  Every per-context fact the
launchers need (shared-memory limits, SM count, occupancy, tensor maps) is
looked up once, so a call costs its argument checks and the launch itself.
This test times back-to-back calls from C (no Python in the loop) on a tiny
batch, for the three launch paths that used to query the runtime on every
call: the split read (occupancy-based split grouping), the single-pass read
and the warp-specialized tcgen05 chunk read (two tensor maps).
"""

import ctypes
import os
import subprocess

import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
DEV = "cuda"
CALLS = 400          # below the launch queue's depth, so the host never waits for the GPU
BOUND_NS = 8000.0    # per call, launch included


@pytest.fixture(scope="module")
def harness(lib, tmp_path_factory):
    libdir = os.path.dirname(lib.LIB_PATH)
    so = str(tmp_path_factory.mktemp("hc") / "libhost_cost.so")
    subprocess.run(["gcc", "-O2", "-shared", "-fPIC", "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, "native", "host_cost.c"), "-o", so, "-L", libdir,
                    "-l:libpa.so", f"-Wl,-rpath,{libdir}"], check=True)
    h = ctypes.CDLL(so)
    p, i, f = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    h.host_cost_decode.restype = ctypes.c_double
    h.host_cost_decode.argtypes = [ctypes.c_int, p, p, p, p, p, i, p, i, i, i, i, i, i, f, i]
    h.host_cost_splitkv.restype = ctypes.c_double
    h.host_cost_splitkv.argtypes = [ctypes.c_int, p, p, p, p, p, p, i, p, i, i, i, i, i, i, f,
                                    i, i, i]
    h.host_cost_chunk.restype = ctypes.c_double
    h.host_cost_chunk.argtypes = [ctypes.c_int, p, p, p, p, p, i, p, i, i, i, i, i, i, i, f, i]
    return h


def _timed(fn):
    fn(50)                       # first calls: module load, per-context lookups
    torch.cuda.synchronize()
    ns = fn(CALLS)
    torch.cuda.synchronize()
    assert ns > 0, f"status {-ns}"
    return ns


def test_split_and_single_pass_reads_cost_little_host_time(lib, harness):
    g = workloads.llama1b(64, batch=1).to(DEV)
    out = torch.empty_like(g.q)
    po = torch.empty((1, 32, 4, 64), device=DEV)
    pl = torch.empty((1, 32, 4), device=DEV)
    args = (g.q.data_ptr(), g.k_pool.data_ptr(), g.v_pool.data_ptr(), g.block_table.data_ptr(),
            g.max_blocks, g.seq_lens.data_ptr(), 1, 32, 8, 64, 16, g.num_pages, g.scale)
    split_ns = _timed(lambda n: harness.host_cost_splitkv(n, po.data_ptr(), pl.data_ptr(), *args,
                                                          1, 4, lib.PA_BF16))
    decode_ns = _timed(lambda n: harness.host_cost_decode(n, out.data_ptr(), *args, lib.PA_BF16))
    print(f"host ns per call: pa_decode_splitkv {split_ns:.0f}, pa_decode {decode_ns:.0f}")
    assert split_ns < BOUND_NS and decode_ns < BOUND_NS


def test_warp_specialized_chunk_read_costs_little_host_time(lib, harness):
    base = workloads.make_batch("hc_chunk", 61, "bf16", [128], 4, 1, 64, 16, 12)
    g = base.to(DEV)
    gen = torch.Generator(device=DEV)
    gen.manual_seed(0)
    q = torch.randn((1, 64, 4, 64), generator=gen, device=DEV).to(torch.bfloat16)  # 256 rows
    out = torch.empty_like(q)
    ns = _timed(lambda n: harness.host_cost_chunk(
        n, out.data_ptr(), q.data_ptr(), g.k_pool.data_ptr(), g.v_pool.data_ptr(),
        g.block_table.data_ptr(), g.max_blocks, g.seq_lens.data_ptr(), 1, 64, 4, 1, 64, 16,
        g.num_pages, g.scale, lib.PA_BF16))
    print(f"host ns per call: pa_decode_chunk (tcgen05, tensor maps) {ns:.0f}")
    assert ns < BOUND_NS
