// Device helpers shared by the kernels: element conversion, cp.async,
// error recording.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace pa {

// Programmatic dependent launch: a kernel launched with the
// programmatic-stream-serialization attribute may start while the kernel
// before it in the stream is finishing; pdl_wait() blocks until that kernel
// has completed and its writes are visible (a no-op when there is none).
// pdl_trigger() lets the next kernel in the stream start its launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Record the first device-side error of a launch (first writer wins).
__device__ __forceinline__ void report_error(int32_t *dev_err, int32_t code) {
  if (dev_err != nullptr) atomicCAS(dev_err, 0, code);
}

// 2^x by the SFU's approximate base-2 exponential (relative error about
// 2^-22; 2^-inf = +0, subnormal results flush to zero).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- 16-byte chunk -> fp32 ------------------------------------------------

template <typename T> struct Elem;

template <> struct Elem<float> {
  static constexpr int kPerChunk = 4;
  __device__ __forceinline__ static void to_f32(const uint4 &c, float *o) {
    o[0] = __uint_as_float(c.x); o[1] = __uint_as_float(c.y);
    o[2] = __uint_as_float(c.z); o[3] = __uint_as_float(c.w);
  }
  __device__ __forceinline__ static float from_f32(float x) { return x; }
  using Storage = float;
};

// bf16 is the upper half of an fp32 bit pattern, so widening is a shift.
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float &lo, float &hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

template <> struct Elem<__nv_bfloat16> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void to_f32(const uint4 &c, float *o) {
    bf16x2_to_f32(c.x, o[0], o[1]); bf16x2_to_f32(c.y, o[2], o[3]);
    bf16x2_to_f32(c.z, o[4], o[5]); bf16x2_to_f32(c.w, o[6], o[7]);
  }
  using Storage = __nv_bfloat16;
};

template <> struct Elem<__half> {
  static constexpr int kPerChunk = 8;
  __device__ __forceinline__ static void to_f32(const uint4 &c, float *o) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 f = __half22float2(h);
      o[2 * i] = f.x; o[2 * i + 1] = f.y;
    }
  }
  using Storage = __half;
};

// fp32 -> storage type, round to nearest even.
template <typename T> __device__ __forceinline__ T cvt_out(float x);
template <> __device__ __forceinline__ float cvt_out<float>(float x) { return x; }
template <> __device__ __forceinline__ __half cvt_out<__half>(float x) { return __float2half_rn(x); }
template <> __device__ __forceinline__ __nv_bfloat16 cvt_out<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// ---- cp.async (16 bytes, L2 only) -----------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Copies 16 bytes when valid, otherwise fills the 16 shared bytes with zeros
// (src-size 0: no global byte is read).
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src, bool valid) {
  const int src_bytes = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}

template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;\n" ::: "memory");
}

}  // namespace pa
