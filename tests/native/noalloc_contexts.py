"""Child process of tests/test_zz_no_alloc.py: pa_decode_splitkv_noalloc in two CUDA
contexts on one device.

The library's fixed partials array is loaded into every context that runs the
library's kernels, at an address of that context.  This script runs the call in the
device's primary context, then in a second context it creates on the same device
(through the driver API, with its own buffers), then in the primary context again,
and saves the three outputs for the parent test to compare with the existing entry
points.  It uses no torch: inputs arrive as NumPy arrays in an .npz file.

usage: noalloc_contexts.py <inputs.npz> <outputs.npz> <libpa.so>
"""

import ctypes
import sys

import numpy as np


def main():
    inp, outp, libpa_path = sys.argv[1:4]
    data = np.load(inp)
    cu = ctypes.CDLL("libcuda.so.1")
    lib = ctypes.CDLL(libpa_path)
    p, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    lib.pa_decode_splitkv_noalloc.restype = ctypes.c_int
    lib.pa_decode_splitkv_noalloc.argtypes = [p, p, p, p, p, i32, p, i32, i32, i32, i32, i32,
                                              i32, f32, i32, ctypes.c_int, p, p]

    def ck(r, what):
        if r != 0:
            raise RuntimeError(f"{what} returned {r}")

    ck(cu.cuInit(0), "cuInit")
    dev = ctypes.c_int(0)
    ck(cu.cuDeviceGet(ctypes.byref(dev), 0), "cuDeviceGet")
    primary = ctypes.c_void_p()
    ck(cu.cuDevicePrimaryCtxRetain(ctypes.byref(primary), dev), "cuDevicePrimaryCtxRetain")

    def run(ctx, case):
        ck(cu.cuCtxSetCurrent(ctx), "cuCtxSetCurrent")
        arrays = {k: np.ascontiguousarray(data[f"{case}_{k}"])
                  for k in ("q", "k_pool", "v_pool", "block_table", "seq_lens")}
        dptr = {}
        for k, a in list(arrays.items()) + [("out", np.empty_like(arrays["q"]))]:
            d = ctypes.c_uint64()
            ck(cu.cuMemAlloc_v2(ctypes.byref(d), ctypes.c_size_t(max(16, a.nbytes))),
               "cuMemAlloc")
            if k != "out":
                ck(cu.cuMemcpyHtoD_v2(d, a.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.c_size_t(a.nbytes)), "cuMemcpyHtoD")
            dptr[k] = d.value
        meta = data[f"{case}_meta"]   # scale, block_size, pages_per_split, dtype code
        q = arrays["q"]
        npg, bs, hkv, d = arrays["k_pool"].shape
        st = lib.pa_decode_splitkv_noalloc(
            dptr["out"], dptr["q"], dptr["k_pool"], dptr["v_pool"], dptr["block_table"],
            arrays["block_table"].shape[1], dptr["seq_lens"], q.shape[0], q.shape[1], hkv, d,
            bs, npg, float(meta[0]), int(meta[2]), int(meta[3]), None, None)
        ck(st, "pa_decode_splitkv_noalloc")
        ck(cu.cuCtxSynchronize(), "cuCtxSynchronize")
        out = np.empty_like(q)
        ck(cu.cuMemcpyDtoH_v2(out.ctypes.data_as(ctypes.c_void_p), ctypes.c_uint64(dptr["out"]),
                              ctypes.c_size_t(out.nbytes)), "cuMemcpyDtoH")
        for v in dptr.values():
            ck(cu.cuMemFree_v2(ctypes.c_uint64(v)), "cuMemFree")
        return out

    cases = [str(c) for c in data["cases"]]
    results = {}
    for c in cases:
        results[f"{c}_primary"] = run(primary, c)
    second = ctypes.c_void_p()
    ck(cu.cuCtxCreate_v2(ctypes.byref(second), 0, dev), "cuCtxCreate")
    for c in cases:
        results[f"{c}_second"] = run(second, c)
    for c in cases:
        results[f"{c}_primary_again"] = run(primary, c)
    ck(cu.cuCtxSetCurrent(primary), "cuCtxSetCurrent")
    ck(cu.cuCtxDestroy_v2(second), "cuCtxDestroy")
    ck(cu.cuDevicePrimaryCtxRelease_v2(dev), "cuDevicePrimaryCtxRelease")
    np.savez(outp, **results)
    print("contexts ok")


if __name__ == "__main__":
    main()
