// Paged decode attention on the CUDA cores (fp32 FMA) for f16/bf16 caches at
// head dims the tensor-core read does not cover (fp32 caches have their own
// read, pa_decode_f32.cu).
//
// One CTA per (sequence, kv head, split).  The CTA walks its token range of
// the block table ("Three Attention Kernels", section "3. Paged KV-cache
// attention": page = block_table[b][p / page_size], row = p % page_size),
// streams K and V rows of its kv head through a 4-stage cp.async ring in
// shared memory, and keeps an online softmax per query head (nanoserve
// "Day 23: the real triton.jit paged-attention kernel": running max and
// sum, accumulator rescaled when the max grows, the score row never
// stored).  Unlike the pages' Triton kernel (one program per query head),
// the whole GQA group of query heads is handled by one CTA, so every K/V
// row is read from HBM once.
//
// Work split inside the CTA: threads form lane groups of TG lanes; a group
// owns one token at a time and each lane owns CPL 16-byte chunks of the
// head dimension.  Scores are lane-partial dot products summed with xor
// shuffles inside the group; P.V needs no communication because the lane
// accumulates exactly the channels it loaded.  Every group keeps its own
// (m, l, acc) over the tokens it saw; the groups are combined once at the
// end through shared memory.  Ragged tails and head dims that are not a
// power of two are handled by predication (zero-filled copies, masked
// scores), never by padding the data.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kTokPerGroup = 4;  // tokens one lane group takes per stage
constexpr int kStages = 4;

template <typename T, int GMAX, int CPL>
__global__ void __launch_bounds__(kThreads)
    decode_simt_kernel(const DecodeParams p, const int nch, const int tg_log2) {
  using E = Elem<T>;
  constexpr int EPC = E::kPerChunk;  // elements in a 16-byte chunk
  constexpr int EPL = EPC * CPL;     // channels one lane owns
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int s_bad;

  const int tg = 1 << tg_log2;
  const int ng = kThreads >> tg_log2;  // lane groups in the CTA
  const int tt = ng * kTokPerGroup;    // tokens per pipeline stage
  const int tid = threadIdx.x;
  const int grp = tid >> tg_log2;
  const int j = tid & (tg - 1);

  const int hkv = p.num_kv_heads;
  const int g = blockIdx.x % hkv;
  const int split = blockIdx.x / hkv;
  const int b = blockIdx.y;
  const int D = p.head_dim;
  const int G = p.group;
  const int bs_log2 = p.block_size_log2;
  const int bs_mask = (1 << bs_log2) - 1;

  if (tid == 0) s_bad = 0;

  // ---- token range of this CTA -------------------------------------------
  int len = p.seq_lens[b];
  const long long cap = static_cast<long long>(p.max_blocks) << bs_log2;
  const bool bad_len = (len < 0) || (static_cast<long long>(len) > cap);
  if (bad_len) {
    if (tid == 0) report_error(p.dev_err, PA_DEV_BAD_SEQ_LEN);
    len = 0;
  }
  int t_begin = 0, t_end = len;
  if (p.pages_per_split > 0) {
    const long long span = static_cast<long long>(p.pages_per_split) << bs_log2;
    const long long lo = static_cast<long long>(split) * span;
    t_begin = static_cast<int>(min(static_cast<long long>(len), lo));
    t_end = static_cast<int>(min(static_cast<long long>(len), lo + span));
  }

  // ---- q of the group's heads, pre-scaled into base-2 score units --------
  float qf[GMAX][EPL];
  {
    const T *qb = static_cast<const T *>(p.q) +
                  (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G) * D;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int chunk = j + c * tg;
        if (h < G && chunk < nch) {
          const uint4 raw = *reinterpret_cast<const uint4 *>(qb + h * D + chunk * EPC);
          E::to_f32(raw, &qf[h][c * EPC]);
#pragma unroll
          for (int e = 0; e < EPC; ++e) qf[h][c * EPC + e] *= p.scale_log2;
        } else {
#pragma unroll
          for (int e = 0; e < EPC; ++e) qf[h][c * EPC + e] = 0.f;
        }
      }
    }
  }

  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  const T *kpool = static_cast<const T *>(p.k_pool);
  const T *vpool = static_cast<const T *>(p.v_pool);
  const int stage_chunks = tt * nch;
  const size_t stage_bytes = static_cast<size_t>(stage_chunks) * 16 * 2;
  __syncthreads();  // s_bad initialised before any loader may set it

  auto load_tile = [&](int it, int stage) {
    const int tok0 = t_begin + it * tt;
    uint4 *ks = reinterpret_cast<uint4 *>(smem + stage * stage_bytes);
    uint4 *vs = ks + stage_chunks;
    for (int idx = tid; idx < stage_chunks; idx += kThreads) {
      const int t = idx / nch;
      const int c = idx - t * nch;
      const int pos = tok0 + t;
      bool valid = pos < t_end;
      const T *ksrc = kpool;
      const T *vsrc = vpool;
      if (valid) {
        const int page = bt_row[pos >> bs_log2];
        if (page < 0 || page >= p.num_pages) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          s_bad = 1;
          valid = false;
        } else {
          const size_t row = (static_cast<size_t>(page) << bs_log2) + (pos & bs_mask);
          const size_t off = (row * hkv + g) * D + static_cast<size_t>(c) * EPC;
          ksrc += off;
          vsrc += off;
        }
      }
      cp_async16(ks + idx, ksrc, valid);
      cp_async16(vs + idx, vsrc, valid);
    }
  };

  const int ntok = t_end - t_begin;
  const int ntiles = ntok > 0 ? (ntok + tt - 1) / tt : 0;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s, s);
    cp_async_commit();
  }

  float m[GMAX], l[GMAX], acc[GMAX][EPL];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[h][e] = 0.f;
  }

  for (int it = 0; it < ntiles; ++it) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nt = it + kStages - 1;
      if (nt < ntiles) load_tile(nt, nt % kStages);
      cp_async_commit();
    }
    const uint4 *ks = reinterpret_cast<const uint4 *>(smem + (it % kStages) * stage_bytes);
    const uint4 *vs = ks + stage_chunks;
    const int tok0 = t_begin + it * tt;

    // scores of this group's tokens (base-2 units)
    float sc[kTokPerGroup][GMAX];
#pragma unroll
    for (int k = 0; k < kTokPerGroup; ++k) {
      const int t = grp + k * ng;
      float kf[EPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int chunk = j + c * tg;
        if (chunk < nch) {
          E::to_f32(ks[t * nch + chunk], &kf[c * EPC]);
        } else {
#pragma unroll
          for (int e = 0; e < EPC; ++e) kf[c * EPC + e] = 0.f;
        }
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qf[h][e], kf[e], dot);
        for (int off = tg >> 1; off > 0; off >>= 1)
          dot += __shfl_xor_sync(0xffffffffu, dot, off);
        sc[k][h] = (tok0 + t < t_end) ? dot : -CUDART_INF_F;
      }
    }

    // online softmax: new running max, rescale, probabilities
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float mt = sc[0][h];
#pragma unroll
      for (int k = 1; k < kTokPerGroup; ++k) mt = fmaxf(mt, sc[k][h]);
      const float mn = fmaxf(m[h], mt);
      if (mn == -CUDART_INF_F) {
#pragma unroll
        for (int k = 0; k < kTokPerGroup; ++k) sc[k][h] = 0.f;
        continue;
      }
      const float alpha = exp2f(m[h] - mn);
      float psum = 0.f;
#pragma unroll
      for (int k = 0; k < kTokPerGroup; ++k) {
        sc[k][h] = exp2f(sc[k][h] - mn);
        psum += sc[k][h];
      }
      l[h] = fmaf(l[h], alpha, psum);
      m[h] = mn;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[h][e] *= alpha;
    }

    // P.V on the channels this lane owns
#pragma unroll
    for (int k = 0; k < kTokPerGroup; ++k) {
      const int t = grp + k * ng;
      float vf[EPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int chunk = j + c * tg;
        if (chunk < nch) {
          E::to_f32(vs[t * nch + chunk], &vf[c * EPC]);
        } else {
#pragma unroll
          for (int e = 0; e < EPC; ++e) vf[c * EPC + e] = 0.f;
        }
      }
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[h][e] = fmaf(sc[k][h], vf[e], acc[h][e]);
      }
    }
  }
  cp_async_wait_all();
  __syncthreads();  // ring no longer read: reuse it for the group combine

  // ---- combine the lane groups ---------------------------------------------
  float *sm_m = reinterpret_cast<float *>(smem);
  float *sm_l = sm_m + ng * GMAX;
  float *sm_acc = sm_l + ng * GMAX;  // [ng][GMAX][D]
  if (j == 0) {
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      sm_m[grp * GMAX + h] = m[h];
      sm_l[grp * GMAX + h] = l[h];
    }
  }
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int chunk = j + c * tg;
      if (h < G && chunk < nch) {
#pragma unroll
        for (int e = 0; e < EPC; ++e)
          sm_acc[(grp * GMAX + h) * D + chunk * EPC + e] = acc[h][c * EPC + e];
      }
    }
  }
  __syncthreads();

  const bool bad = bad_len || (s_bad != 0);
  const bool is_split = p.pages_per_split > 0;
  for (int o = tid; o < G * D; o += kThreads) {
    const int h = o / D;
    const int e = o - h * D;
    float M = -CUDART_INF_F;
    for (int gi = 0; gi < ng; ++gi) M = fmaxf(M, sm_m[gi * GMAX + h]);
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
      for (int gi = 0; gi < ng; ++gi) {
        const float w = exp2f(sm_m[gi * GMAX + h] - M);
        L = fmaf(sm_l[gi * GMAX + h], w, L);
        O = fmaf(sm_acc[(gi * GMAX + h) * D + e], w, O);
      }
    }
    const bool empty = bad || (M == -CUDART_INF_F);
    const float res = empty ? 0.f : O / L;
    const size_t qh = static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G + h;
    if (is_split) {
      const size_t row = qh * p.num_splits + split;
      p.partial_out[row * D + e] = res;
      if (e == 0)
        p.partial_lse[row] = empty ? -CUDART_INF_F : (M + log2f(L)) * 0.69314718055994531f;
    } else {
      static_cast<T *>(p.out)[qh * D + e] = cvt_out<T>(res);
    }
  }
}

int ceil_log2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

template <typename T, int GMAX, int CPL>
cudaError_t launch_shape(const DecodeParams &p, int nch, int tg_log2, cudaStream_t stream) {
  const int ng = kThreads >> tg_log2;
  const int tt = ng * kTokPerGroup;
  const size_t ring = static_cast<size_t>(kStages) * tt * nch * 16 * 2;
  const size_t combine = static_cast<size_t>(ng) * GMAX * (2 + p.head_dim) * sizeof(float);
  const size_t smem = ring > combine ? ring : combine;
  auto kern = decode_simt_kernel<T, GMAX, CPL>;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  dim3 grid(p.num_splits * p.num_kv_heads, p.num_seqs);
  kern<<<grid, kThreads, smem, stream>>>(p, nch, tg_log2);
  return cudaGetLastError();
}

template <typename T, int CPL>
cudaError_t launch_group(const DecodeParams &p, int nch, int tg_log2, cudaStream_t stream) {
  if (p.group <= 1) return launch_shape<T, 1, CPL>(p, nch, tg_log2, stream);
  if (p.group <= 2) return launch_shape<T, 2, CPL>(p, nch, tg_log2, stream);
  if (p.group <= 4) return launch_shape<T, 4, CPL>(p, nch, tg_log2, stream);
  return launch_shape<T, 8, CPL>(p, nch, tg_log2, stream);
}

template <typename T>
cudaError_t launch_typed(const DecodeParams &p, cudaStream_t stream) {
  const int nch = p.head_dim * static_cast<int>(sizeof(T)) / 16;  // <= 32 at head_dim <= 256
  return launch_group<T, 1>(p, nch, ceil_log2(nch), stream);
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream) {
  switch (dtype) {
    case PA_F16: return launch_typed<__half>(p, stream);
    case PA_BF16: return launch_typed<__nv_bfloat16>(p, stream);
    case PA_F32: break;  // fp32 caches: launch_decode_f32
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
