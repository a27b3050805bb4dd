// Cross-split combine of split-KV partials.
//
// "Three Attention Kernels", section "2. Split-KV flash-decoding": after
// every split reduced its slice, the outputs are combined with weights
// exp(lse_s - max lse), normalised by their sum.  One warp per (sequence,
// query head) row: lanes stride over the splits for the max and the
// weights, then over the head dimension (coalesced) for the weighted sum.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxPerLane = 8;  // head_dim <= 256

template <typename T>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeParams p) {
  pdl_wait();  // the partials come from the split read just before
  const int row = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.rows) return;
  const int S = p.num_splits;
  const int D = p.head_dim;
  const float *lse = p.partial_lse + static_cast<size_t>(row) * S;
  const float *po = p.partial_out + static_cast<size_t>(row) * S * D;
  T *out = static_cast<T *>(p.out) + static_cast<size_t>(row) * D;

  float M = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse[s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (M == -CUDART_INF_F) {
    for (int e = lane; e < D; e += 32) out[e] = cvt_out<T>(0.f);
    return;
  }

  float o[kMaxPerLane];
#pragma unroll
  for (int k = 0; k < kMaxPerLane; ++k) o[k] = 0.f;
  float wsum = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const float w_lane = (s0 + lane < S) ? expf(lse[s0 + lane] - M) : 0.f;
    wsum += w_lane;
    const int n = min(32, S - s0);
    for (int i = 0; i < n; ++i) {
      const float w = __shfl_sync(0xffffffffu, w_lane, i);
      if (w == 0.f) continue;  // empty split: carries no weight
      const float *src = po + static_cast<size_t>(s0 + i) * D;
#pragma unroll
      for (int k = 0; k < kMaxPerLane; ++k) {
        const int e = lane + 32 * k;
        if (e < D) o[k] = fmaf(w, src[e], o[k]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  const float inv = 1.f / wsum;
#pragma unroll
  for (int k = 0; k < kMaxPerLane; ++k) {
    const int e = lane + 32 * k;
    if (e < D) out[e] = cvt_out<T>(o[k] * inv);
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, pa_dtype dtype, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((p.rows + kWarps - 1) / kWarps);
  switch (dtype) {
    case PA_F32: return launch_pdl(merge_kernel<float>, dim3(blocks), dim3(kThreads), 0, stream, p);
    case PA_F16: return launch_pdl(merge_kernel<__half>, dim3(blocks), dim3(kThreads), 0, stream, p);
    case PA_BF16:
      return launch_pdl(merge_kernel<__nv_bfloat16>, dim3(blocks), dim3(kThreads), 0, stream, p);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
