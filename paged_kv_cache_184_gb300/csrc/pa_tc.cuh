// tcgen05 building blocks shared by the chunked-read kernels: shared-memory
// and instruction descriptors, the MMA forms, commit and bounded mbarrier
// waits, tensor-memory loads and stores, 16-bit packing, and the 128-byte
// swizzle of the K-major / MN-major tiles the tensor core reads.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "pa_common.cuh"  // ex2_approx

namespace pa {
namespace tc {

// A wait on an mbarrier gives up (and the kernel reports PA_DEV_TIMEOUT
// instead of hanging) after about a second, or after kSpinLimit polls,
// whichever comes first.  A poll that finds the phase incomplete may suspend
// the thread for microseconds, so the time bound is the one that acts.
constexpr uint32_t kSpinLimit = 1u << 26;
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version of this architecture
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulate, A/B element type,
// A K-major, B K-major or MN-major, N and M.
template <typename T>
__host__ __device__ constexpr uint32_t idesc(int m, int n, bool b_mn_major, bool negate_a) {
  const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((negate_a ? 1u : 0u) << 13) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t id,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(da), "l"(db), "r"(id), "r"(accumulate));
}

// The same product with A read from tensor memory (128 lanes x 8 columns of
// packed 16-bit pairs per 16-wide K step) instead of a shared-memory descriptor.
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t db,
                                           uint32_t id, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(db), "r"(id), "r"(accumulate));
}

__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   mbar)
               : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// arrive on `bar` and expect `bytes` more from bulk copies before its phase completes
__device__ __forceinline__ void mbar_arrive_expect(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 2D tile copy through a tensor map (128-byte swizzle), counted on `bar`;
// x (elements) is a multiple of 64, so x * 2 bytes is 16-byte aligned
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Wait for the given phase of an mbarrier; false once the bounds above are
// reached.  Each poll passes a 20 ns suspend hint (measured a few per cent
// faster than the default limit).
__device__ __forceinline__ bool wait_phase(uint32_t mbar, uint32_t phase) {
  uint64_t t0 = 0;
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(done)
        : "r"(mbar), "r"(phase)
        : "memory");
    if (done) return true;
    if (it == 0) {
      t0 = global_ns();
    } else if ((it & 15) == 0 && global_ns() - t0 > kWaitLimitNs) {
      return false;
    }
  }
  return false;
}

// The wait for tcgen05.ld / tcgen05.st, with 32 registers tied to it: the
// registers a load writes are read only after the wait, and the registers a
// store reads keep their values (are not reused) until the wait.
#define PA_TIE32(q)                                                                        \
  "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]), "+r"(q[4]), "+r"(q[5]), "+r"(q[6]),      \
      "+r"(q[7]), "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]), "+r"(q[12]),           \
      "+r"(q[13]), "+r"(q[14]), "+r"(q[15]), "+r"(q[16]), "+r"(q[17]), "+r"(q[18]),        \
      "+r"(q[19]), "+r"(q[20]), "+r"(q[21]), "+r"(q[22]), "+r"(q[23]), "+r"(q[24]),        \
      "+r"(q[25]), "+r"(q[26]), "+r"(q[27]), "+r"(q[28]), "+r"(q[29]), "+r"(q[30]),        \
      "+r"(q[31])

__device__ __forceinline__ void wait_ld_tied(uint32_t *q) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PA_TIE32(q)::"memory");
}

__device__ __forceinline__ void wait_st_tied(uint32_t *q) {
  asm volatile("tcgen05.wait::st.sync.aligned;" : PA_TIE32(q)::"memory");
}

__device__ __forceinline__ void tie32(uint32_t *q) { asm volatile("" : PA_TIE32(q)); }

#define PA_TIE16(q)                                                                        \
  "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]), "+r"(q[4]), "+r"(q[5]), "+r"(q[6]),      \
      "+r"(q[7]), "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]), "+r"(q[12]),           \
      "+r"(q[13]), "+r"(q[14]), "+r"(q[15])

__device__ __forceinline__ void wait_st_tied16(uint32_t *q) {
  asm volatile("tcgen05.wait::st.sync.aligned;" : PA_TIE16(q)::"memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  wait_ld_tied(r);
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 64 consecutive columns of this warp's 32 lanes: both loads in flight, one wait
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float *v) {
  uint32_t r[64];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t *q = r + 32 * h;
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
          "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]),
          "=r"(q[14]), "=r"(q[15]), "=r"(q[16]), "=r"(q[17]), "=r"(q[18]), "=r"(q[19]),
          "=r"(q[20]), "=r"(q[21]), "=r"(q[22]), "=r"(q[23]), "=r"(q[24]), "=r"(q[25]),
          "=r"(q[26]), "=r"(q[27]), "=r"(q[28]), "=r"(q[29]), "=r"(q[30]), "=r"(q[31])
        : "r"(taddr + 32 * h));
  }
  wait_ld_tied(r);
  tie32(r + 32);  // after the wait, too
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]),
      "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]), "f"(v[13]), "f"(v[14]),
      "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]),
      "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]),
      "f"(v[29]), "f"(v[30]), "f"(v[31]));
  uint32_t q[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) q[j] = __float_as_uint(v[j]);
  wait_st_tied(q);
}

__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31]));
  uint32_t q[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) q[j] = v[j];
  wait_st_tied(q);
}

// 16 consecutive columns of this warp's 32 lanes into 16 words
__device__ __forceinline__ void tmem_ld16u(uint32_t taddr, uint32_t *q) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(q[0]), "=r"(q[1]), "=r"(q[2]), "=r"(q[3]), "=r"(q[4]), "=r"(q[5]), "=r"(q[6]),
        "=r"(q[7]), "=r"(q[8]), "=r"(q[9]), "=r"(q[10]), "=r"(q[11]), "=r"(q[12]), "=r"(q[13]),
        "=r"(q[14]), "=r"(q[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" : PA_TIE16(q)::"memory");
}

// 16 consecutive columns of this warp's 32 lanes from 16 packed words
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]));
  uint32_t q[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) q[j] = v[j];
  wait_st_tied16(q);
}

template <typename T> struct Pack2;
template <> struct Pack2<__nv_bfloat16> {
  __device__ __forceinline__ static uint32_t run(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <> struct Pack2<__half> {
  __device__ __forceinline__ static uint32_t run(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

// byte offset of 16-byte chunk `chunk` of row `row` in a [kb][rows][128 B] swizzled tile
__device__ __forceinline__ uint32_t sw_off(int row, int chunk, int rows) {
  return (chunk >> 3) * rows * 128 + row * 128 + (((chunk & 7) ^ (row & 7)) << 4);
}

// ---- per-row softmax pieces on 64 scores (one row per thread) -------------
// Paired fp32 arithmetic (f32x2) and the three-input max halve the issue
// slots of the row max, the exponent arguments and the row sum; the
// exponentials themselves stay one ex2.approx per score.

__device__ __forceinline__ uint64_t pack_f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

__device__ __forceinline__ void unpack_f2(uint64_t v, float &a, float &b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// max of s[0..63] (-inf when every score is masked)
__device__ __forceinline__ float row_max64(const float *s) {
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float m = max3(s[i], s[i + 8], s[i + 16]);
    m = max3(m, s[i + 24], s[i + 32]);
    m = max3(m, s[i + 40], s[i + 48]);
    r[i] = fmaxf(m, s[i + 56]);
  }
  return max3(max3(r[0], r[1], r[2]), max3(r[3], r[4], r[5]), fmaxf(r[6], r[7]));
}

// s[c] <- 2^(s[c] * sl2 - mu) in place (a masked -inf gives 0); returns the sum
__device__ __forceinline__ float row_exp64(float *s, float sl2, float mu) {
  const uint64_t scale = pack_f2(sl2, sl2), shift = pack_f2(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    uint64_t x;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(pack_f2(s[2 * c], s[2 * c + 1])),
        "l"(scale), "l"(shift));
    float a, b;
    unpack_f2(x, a, b);
    a = ex2_approx(a);
    b = ex2_approx(b);
    s[2 * c] = a;
    s[2 * c + 1] = b;
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[c & 3]) : "l"(pack_f2(a, b)));
  }
  float t[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack_f2(acc[i], t[2 * i], t[2 * i + 1]);
  return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
}

// The same two pieces on N scores (N a multiple of 8).
template <int N>
__device__ __forceinline__ float row_max_n(const float *s) {
  float r[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float m = s[i];
    int c = i + 8;
#pragma unroll
    for (; c + 8 < N; c += 16) m = max3(m, s[c], s[c + 8]);
    if (c < N) m = fmaxf(m, s[c]);
    r[i] = m;
  }
  return max3(max3(r[0], r[1], r[2]), max3(r[3], r[4], r[5]), fmaxf(r[6], r[7]));
}

template <int N>
__device__ __forceinline__ float row_exp_n(float *s, float sl2, float mu) {
  const uint64_t scale = pack_f2(sl2, sl2), shift = pack_f2(-mu, -mu);
  uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
  for (int c = 0; c < N / 2; ++c) {
    uint64_t x;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(x) : "l"(pack_f2(s[2 * c], s[2 * c + 1])),
        "l"(scale), "l"(shift));
    float a, b;
    unpack_f2(x, a, b);
    a = ex2_approx(a);
    b = ex2_approx(b);
    s[2 * c] = a;
    s[2 * c + 1] = b;
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc[c & 3]) : "l"(pack_f2(a, b)));
  }
  float t[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack_f2(acc[i], t[2 * i], t[2 * i + 1]);
  return ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
}

}  // namespace tc
}  // namespace pa
