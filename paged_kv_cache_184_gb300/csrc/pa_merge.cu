// Cross-split combine of split-KV partials.
//
// "Three Attention Kernels", section "2. Split-KV flash-decoding": after
// every split reduced its slice, the outputs are combined with weights
// exp(lse_s - max lse), normalised by their sum.
//
// One CTA per (sequence, query head) row.  The row's partials are S rows of
// D floats; the CTA's threads form groups of D/4 threads, each thread one
// float4 column, each group every G-th split, so every pass of the loop
// issues a coalesced D*4-byte read per group and several passes are in
// flight at once.  Groups are summed through shared memory at the end.
// Empty splits (lse -inf, weight 0) are skipped without reading them.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kUnroll = 4;

template <typename T>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeParams p) {
  __shared__ float4 s_acc[kThreads];
  __shared__ float s_red[kThreads / 32];
  __shared__ float s_wsum[kThreads];
  pdl_wait();  // the partials come from the split read just before
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int S = p.num_splits;
  const int D = p.head_dim;
  const int cols = D / 4;                // float4 columns
  const int groups = kThreads / cols;    // split groups
  const int grp = tid / cols;
  const int col = tid - grp * cols;
  const bool active = grp < groups;
  const float *lse = p.partial_lse + static_cast<size_t>(row) * S;
  const float4 *po =
      reinterpret_cast<const float4 *>(p.partial_out + static_cast<size_t>(row) * S * D);
  T *out = static_cast<T *>(p.out) + static_cast<size_t>(row) * D;

  // max lse over the splits
  float M = -CUDART_INF_F;
  for (int s = tid; s < S; s += kThreads) M = fmaxf(M, __ldg(lse + s));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if ((tid & 31) == 0) s_red[tid >> 5] = M;
  __syncthreads();
  M = s_red[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) M = fmaxf(M, s_red[w]);
  if (M == -CUDART_INF_F) {  // every split empty
    for (int d = tid; d < D; d += kThreads) out[d] = cvt_out<T>(0.f);
    return;
  }

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (active) {
    for (int s0 = grp; s0 < S; s0 += groups * kUnroll) {
      float w[kUnroll];
      float4 v[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int s = s0 + u * groups;
        w[u] = s < S ? expf(__ldg(lse + s) - M) : 0.f;
        v[u] = w[u] != 0.f ? __ldg(po + static_cast<size_t>(s) * cols + col)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
        wsum += w[u];
      }
    }
  }
  s_acc[tid] = acc;
  s_wsum[tid] = (active && col == 0) ? wsum : 0.f;
  __syncthreads();
  if (tid < cols) {
    float4 t = s_acc[tid];
    float W = s_wsum[0];
    for (int gi = 1; gi < groups; ++gi) {
      const float4 o = s_acc[gi * cols + tid];
      t.x += o.x;
      t.y += o.y;
      t.z += o.z;
      t.w += o.w;
      W += s_wsum[gi * cols];
    }
    const float inv = 1.f / W;
    out[4 * tid] = cvt_out<T>(t.x * inv);
    out[4 * tid + 1] = cvt_out<T>(t.y * inv);
    out[4 * tid + 2] = cvt_out<T>(t.z * inv);
    out[4 * tid + 3] = cvt_out<T>(t.w * inv);
  }
}

}  // namespace

cudaError_t launch_merge(const MergeParams &p, pa_dtype dtype, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.rows));
  switch (dtype) {
    case PA_F32: return launch_pdl(merge_kernel<float>, grid, dim3(kThreads), 0, stream, p);
    case PA_F16: return launch_pdl(merge_kernel<__half>, grid, dim3(kThreads), 0, stream, p);
    case PA_BF16:
      return launch_pdl(merge_kernel<__nv_bfloat16>, grid, dim3(kThreads), 0, stream, p);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
