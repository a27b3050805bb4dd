// Paged decode attention for fp32 caches, on the CUDA cores (fp32 FMA).
//
// Same contract as the other reads: one CTA per (sequence, kv head, split),
// the block-table walk of "Three Attention Kernels" section "3. Paged
// KV-cache attention", and the online softmax of nanoserve "Day 23: the
// real triton.jit paged-attention kernel" (a running reference max and sum,
// the score row never stored), with the whole GQA group in one CTA so that
// every K/V row leaves HBM once.  fp32 needs fp32 products (the 1e-5
// tolerance rules out tf32 tensor cores), so the work is laid out to keep
// the CUDA cores busy with FMAs rather than shuffles:
//
//   scores   a warp tile is 16 tokens; lanes t and t + 16 each dot half of
//            token t's K row with every head of the group (q from shared
//            memory as broadcasts), and one xor shuffle joins the halves
//   softmax  per head, a warp-wide reference max that moves only when a
//            score passes it by more than 2^8 (then O and l are rescaled)
//   P.V      lane L owns channel pairs L, L + 32, ...; the tile's
//            probabilities go through shared memory and are read as
//            broadcasts, V rows as consecutive 8-byte words
//
// Each warp streams every kWarps-th tile through its own cp.async ring (no
// CTA barrier in the loop); K rows are stored with a pitch of head_dim + 4
// floats so that the 16 lanes reading 16 different rows hit different banks.
// The warps' states are combined once at the end.  Tokens past the range
// are zero-filled by the copy and masked to -inf.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kTok = 16;          // tokens per warp tile
constexpr int kMaxThreads = 128;
constexpr float kLazyLog2 = 8.f;  // the reference moves when a score passes it by 2^8

// Shape per head-dim bucket: NP channel pairs per lane (head_dim <= 64 NP), warps
// per CTA and ring stages per warp.  Shared memory per CTA (group 8): 105 KB at
// head_dim 64 (two CTAs per SM), 139 KB at 128, 141 KB at 256.
#ifndef PA_F32_STAGES_D64  // ring stages per warp at head_dim <= 64
#define PA_F32_STAGES_D64 3
#endif

template <int NP>
struct F32Shape {
  static constexpr int kWarps = NP <= 2 ? 4 : 2;
  static constexpr int kStages = NP == 1 ? PA_F32_STAGES_D64 : 2;
};

template <int NP>
size_t f32_smem(int d, int group_max) {
  using S = F32Shape<NP>;
  const size_t q = static_cast<size_t>(group_max) * d;
  const size_t probs = static_cast<size_t>(S::kWarps) * kTok * group_max;
  const size_t ring = static_cast<size_t>(S::kWarps) * S::kStages * kTok * ((d + 4) + d);
  const size_t combine = static_cast<size_t>(S::kWarps) * group_max * (d + 2);
  return (q + probs + (ring > combine ? ring : combine)) * sizeof(float);
}

// GMAX: group size bound (1, 2, 4, 8); NP: channel pairs per lane; DT: the head dim
// when it is fixed at compile time (32, 64, 128, 256: index math by shifts, loops
// unrolled), else 0 (read from the parameters).
template <int GMAX, int NP, int DT>
__global__ void __launch_bounds__(kMaxThreads) decode_f32_kernel(const DecodeParams p) {
  constexpr int stages = F32Shape<NP>::kStages;
  extern __shared__ __align__(16) float sm[];
  __shared__ unsigned s_bad;

  const int nwarps = blockDim.x >> 5;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tok = lane & (kTok - 1), half = lane >> 4;
  const int D = DT > 0 ? DT : p.head_dim, PK = D + 4, nch = D >> 2;
  const int G = p.group;
  const int hkv = p.num_kv_heads;
  const int g = blockIdx.x % hkv;
  const int split = blockIdx.x / hkv;
  const int b = blockIdx.y;
  const int bs_log2 = p.block_size_log2, bs_mask = (1 << bs_log2) - 1;
  const int tile_f = kTok * (PK + D);  // floats of one stage: K rows, then V rows

  float *q_s = sm;                                   // [GMAX][D], scaled to base-2 units
  float *p_s = q_s + GMAX * D;                       // [warps][kTok][GMAX]
  float *ring = p_s + nwarps * kTok * GMAX;          // [warps][stages][tile_f]
  float *my_ring = ring + static_cast<size_t>(warp) * stages * tile_f;
  float *my_p = p_s + warp * kTok * GMAX;

  if (tid == 0) s_bad = 0u;
  pdl_wait();

  // ---- token range of this CTA -------------------------------------------
  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  int len = __ldg(p.seq_lens + b);
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

  // ---- q of the group into shared memory (scale * log2 e folded in) -------
  {
    const float *qrow = static_cast<const float *>(p.q) +
                        (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G) * D;
    for (int i = tid; i < GMAX * D; i += blockDim.x)
      q_s[i] = i < G * D ? __ldg(qrow + i) * p.scale_log2 : 0.f;
  }
  __syncthreads();  // q and s_bad ready

  const int ntok = t_end - t_begin;
  const int ntiles = ntok > 0 ? (ntok + kTok - 1) / kTok : 0;
  const int my_tiles = ntiles > warp ? (ntiles - warp + nwarps - 1) / nwarps : 0;
  const float *kpool = static_cast<const float *>(p.k_pool);
  const float *vpool = static_cast<const float *>(p.v_pool);

  // page id of token `tok` of this warp's i-th tile (-1 past the end)
  auto fetch_pid = [&](int i) -> int {
    const int pos = t_begin + (warp + i * nwarps) * kTok + tok;
    return (i < my_tiles && pos < t_end) ? __ldg(bt_row + (pos >> bs_log2)) : -1;
  };
  // copies of this warp's i-th tile into `stage`; lane t < 16 holds token t's page
  auto load_tile = [&](int i, int stage, int pid) {
    const int tok0 = t_begin + (warp + i * nwarps) * kTok;
    float *ks = my_ring + stage * tile_f;
    float *vs = ks + kTok * PK;
    // every lane runs every pass (the shuffle needs the whole warp); a lane past
    // the tile's last chunk (16 * chunks need not be a multiple of 32) copies nothing
    for (int base = 0; base < kTok * nch; base += 32) {
      const int idx = base + lane;
      const bool in_tile = idx < kTok * nch;
      const int row = in_tile ? idx / nch : kTok - 1;
      const int c = idx - row * nch;
      const int pos = tok0 + row;
      const int page = __shfl_sync(0xffffffffu, pid, row);
      if (!in_tile) continue;
      bool valid = pos < t_end;
      const float *ksrc = kpool, *vsrc = vpool;
      if (valid) {
        if (page < 0 || page >= p.num_pages) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          s_bad = 1u;
          valid = false;
        } else {
          const size_t prow = (static_cast<size_t>(page) << bs_log2) + (pos & bs_mask);
          const size_t off = (prow * hkv + g) * D + c * 4;
          ksrc += off;
          vsrc += off;
        }
      }
      cp_async16(ks + row * PK + c * 4, ksrc, valid);
      cp_async16(vs + row * D + c * 4, vsrc, valid);
    }
  };

  int pid_pre = fetch_pid(0);
  for (int s = 0; s < stages - 1; ++s) {
    const int pid_next = fetch_pid(s + 1);
    if (s < my_tiles) load_tile(s, s, pid_pre);
    cp_async_commit();
    pid_pre = pid_next;
  }

  float m[GMAX], l[GMAX], acc[GMAX][NP][2];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    m[h] = -CUDART_INF_F;
    l[h] = 0.f;
#pragma unroll
    for (int i = 0; i < NP; ++i) acc[h][i][0] = acc[h][i][1] = 0.f;
  }
  // this lane's half of a K row: chunks [c0, c1)
  const int c0 = half ? (nch + 1) >> 1 : 0;
  const int c1 = half ? nch : (nch + 1) >> 1;

  for (int i = 0; i < my_tiles; ++i) {
    // the stage of tile i - 1 is free once every lane is past it; a 2-stage ring
    // refills it before waiting for tile i (two tiles in flight during the wait)
    if constexpr (stages > 2) cp_async_wait<stages - 2>();
    __syncwarp();
    {
      const int ni = i + stages - 1;
      if (ni < my_tiles) {
        load_tile(ni, ni % stages, pid_pre);
        pid_pre = fetch_pid(ni + 1);
      }
      cp_async_commit();
    }
    if constexpr (stages <= 2) {
      cp_async_wait<stages - 1>();
      __syncwarp();
    }
    const float *ks = my_ring + (i % stages) * tile_f;
    const float *vs = ks + kTok * PK;
    const int tok0 = t_begin + (warp + i * nwarps) * kTok;

    // scores: this lane's half of token `tok` against every head
    float s[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) s[h] = 0.f;
    const float *krow = ks + tok * PK;
    auto dot_chunk = [&](int c) {
      const float4 k4 = *reinterpret_cast<const float4 *>(krow + c * 4);
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        const float4 q4 = *reinterpret_cast<const float4 *>(q_s + h * D + c * 4);
        s[h] = fmaf(q4.x, k4.x, fmaf(q4.y, k4.y, fmaf(q4.z, k4.z, fmaf(q4.w, k4.w, s[h]))));
      }
    };
    if constexpr (DT > 0) {  // the two halves are DT / 8 chunks each
#pragma unroll
      for (int k = 0; k < DT / 8; ++k) dot_chunk(half * (DT / 8) + k);
    } else {
      for (int c = c0; c < c1; ++c) dot_chunk(c);
    }
    const bool valid = tok0 + tok < t_end;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      s[h] += __shfl_xor_sync(0xffffffffu, s[h], 16);  // the other half of the row
      if (!valid) s[h] = -CUDART_INF_F;
    }

    // online softmax with a lazily moved reference; probabilities to shared memory
    __syncwarp();  // the previous tile's probabilities have been read
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float mx = s[h];
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      if (mx > m[h] + kLazyLog2) {  // warp-uniform
        const float a = m[h] == -CUDART_INF_F ? 0.f : ex2_approx(m[h] - mx);
        m[h] = mx;
        l[h] *= a;
#pragma unroll
        for (int i2 = 0; i2 < NP; ++i2) {
          acc[h][i2][0] *= a;
          acc[h][i2][1] *= a;
        }
      }
      const float pr = ex2_approx(s[h] - (m[h] == -CUDART_INF_F ? 0.f : m[h]));  // masked: 0
      l[h] += half ? 0.f : pr;
      if (half == 0) my_p[tok * GMAX + h] = pr;
    }
    __syncwarp();

    // P.V on this lane's channel pairs
#pragma unroll 8
    for (int t = 0; t < kTok; ++t) {
      float pt[GMAX];
      if constexpr (GMAX >= 4) {
#pragma unroll
        for (int h = 0; h < GMAX; h += 4) {
          const float4 v4 = *reinterpret_cast<const float4 *>(my_p + t * GMAX + h);
          pt[h] = v4.x;
          pt[h + 1] = v4.y;
          pt[h + 2] = v4.z;
          pt[h + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < GMAX; ++h) pt[h] = my_p[t * GMAX + h];
      }
#pragma unroll
      for (int i2 = 0; i2 < NP; ++i2) {
        const int pair = lane + 32 * i2;
        if (2 * pair < D) {
          const float2 v = *reinterpret_cast<const float2 *>(vs + t * D + 2 * pair);
#pragma unroll
          for (int h = 0; h < GMAX; ++h) {
            acc[h][i2][0] = fmaf(pt[h], v.x, acc[h][i2][0]);
            acc[h][i2][1] = fmaf(pt[h], v.y, acc[h][i2][1]);
          }
        }
      }
    }
  }
  cp_async_wait_all();
  pdl_trigger();  // the merge (or the next read) may start launching
  // the lanes' partial sums of l (lanes 0-15 each counted their own tokens)
#pragma unroll
  for (int h = 0; h < GMAX; ++h)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
  __syncthreads();  // every warp is done with its ring: reuse it for the combine

  float *sm_m = ring;                    // [warps][GMAX]
  float *sm_l = sm_m + nwarps * GMAX;    // [warps][GMAX]
  float *sm_o = sm_l + nwarps * GMAX;    // [warps][GMAX][D]
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    if (lane == 0) {
      sm_m[warp * GMAX + h] = m[h];
      sm_l[warp * GMAX + h] = l[h];
    }
#pragma unroll
    for (int i2 = 0; i2 < NP; ++i2) {
      const int pair = lane + 32 * i2;
      if (2 * pair < D) {
        sm_o[(warp * GMAX + h) * D + 2 * pair] = acc[h][i2][0];
        sm_o[(warp * GMAX + h) * D + 2 * pair + 1] = acc[h][i2][1];
      }
    }
  }
  __syncthreads();

  const bool bad = bad_len || (s_bad != 0u);
  const bool is_split = p.pages_per_split > 0;
  for (int idx = tid; idx < G * D; idx += blockDim.x) {
    const int h = idx / D;
    const int d = idx - h * D;
    float Mx = -CUDART_INF_F;
    for (int w = 0; w < nwarps; ++w) Mx = fmaxf(Mx, sm_m[w * GMAX + h]);
    float L = 0.f, O = 0.f;
    if (Mx != -CUDART_INF_F) {
      for (int w = 0; w < nwarps; ++w) {
        const float wgt = exp2f(sm_m[w * GMAX + h] - Mx);
        L = fmaf(sm_l[w * GMAX + h], wgt, L);
        O = fmaf(sm_o[(w * GMAX + h) * D + d], wgt, O);
      }
    }
    const bool empty = bad || (Mx == -CUDART_INF_F);
    const float res = empty ? 0.f : O / L;
    const size_t qh = static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G + h;
    if (is_split) {
      const size_t row = qh * p.num_splits + split;
      p.partial_out[row * D + d] = res;
      if (d == 0)
        p.partial_lse[row] = empty ? -CUDART_INF_F : (Mx + log2f(L)) * 0.69314718055994531f;
    } else {
      static_cast<float *>(p.out)[qh * D + d] = res;
    }
  }
}

template <int GMAX, int NP, int DT>
cudaError_t launch_np(const DecodeParams &p, cudaStream_t stream) {
  const int smem = static_cast<int>(f32_smem<NP>(p.head_dim, GMAX));
  auto kern = decode_f32_kernel<GMAX, NP, DT>;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  dim3 grid(p.num_splits * p.num_kv_heads, p.num_seqs);
  return launch_pdl(kern, grid, dim3(F32Shape<NP>::kWarps * 32), smem, stream, p);
}

template <int GMAX>
cudaError_t launch_g(const DecodeParams &p, cudaStream_t stream) {
  switch (p.head_dim) {
    case 32: return launch_np<GMAX, 1, 32>(p, stream);
    case 64: return launch_np<GMAX, 1, 64>(p, stream);
    case 128: return launch_np<GMAX, 2, 128>(p, stream);
    case 256: return launch_np<GMAX, 4, 256>(p, stream);
  }
  if (p.head_dim <= 64) return launch_np<GMAX, 1, 0>(p, stream);
  if (p.head_dim <= 128) return launch_np<GMAX, 2, 0>(p, stream);
  return launch_np<GMAX, 4, 0>(p, stream);
}

}  // namespace

// fp32 caches, head_dim a multiple of 4 up to 256, groups of up to 8.
cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t stream) {
  if (p.group <= 1) return launch_g<1>(p, stream);
  if (p.group <= 2) return launch_g<2>(p, stream);
  if (p.group <= 4) return launch_g<4>(p, stream);
  return launch_g<8>(p, stream);
}

}  // namespace pa
