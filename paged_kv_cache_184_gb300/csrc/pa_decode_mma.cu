// Paged decode attention on the tensor cores (mma.sync m16n8k16), f16/bf16.
//
// Same contract as the CUDA-core read: one CTA per (sequence, kv head,
// split); the block-table walk and the online softmax follow
// "Three Attention Kernels" section "3. Paged KV-cache attention" and
// nanoserve "Day 23: the real triton.jit paged-attention kernel".  What is
// different is how one 16-token tile is reduced.  The tile is the M side of
// two small matrix products, the GQA group of query heads is the N side:
//
//   S^T [16 tokens x 8 heads] = K_tile [16 x D] . Q^T [D x 8 heads]
//   O^T [D x 8 heads]        += V_tile^T [D x 16] . P^T [16 x 8 heads]
//
// K feeds the first product through ldmatrix, V the second through
// ldmatrix.trans; the probabilities P^T leave the first product's
// accumulators and enter the second as a B operand after one movmatrix
// transpose per 8x8 block, so scores never touch shared memory.  A group
// of up to 8 heads fills one n8 tile, up to 16 heads two.
//
// Every warp owns every NW-th tile of the CTA's token range and streams it
// through its own NS-stage cp.async ring (no CTA barrier in the main loop);
// the warps' (m, l, O) states are combined at the end of every split.  In
// the split read a CTA may cover several consecutive splits of one
// (sequence, kv head): the warps' copies run on across split boundaries
// while each finished split is combined in a separate area, so one
// pipeline ramp serves all of them and the whole grid fits one wave.  Rows are stored
// with a 16-byte-chunk XOR swizzle so that ldmatrix is bank-conflict free.
// Tokens past the end of the range are zero-filled by the copy and masked
// to -inf in the scores.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Ring shape: warps per CTA and copy stages per warp (smem per CTA is
// warps x stages x 2 tiles).  At head_dim 64, 4 warps x 3 stages = 48 KB
// keeps 4 CTAs per SM, so 64 sequences x 8 kv heads run in one wave; at
// head_dim 128, 2 stages (64 KB, 3 CTAs per SM) measured faster than 3.
#ifndef PA_MMA_WARPS
#define PA_MMA_WARPS 4
#endif
#ifndef PA_MMA_STAGES_D64   // head_dim <= 64
#define PA_MMA_STAGES_D64 3
#endif
#ifndef PA_MMA_STAGES_D128  // 64 < head_dim <= 128
#define PA_MMA_STAGES_D128 2
#endif

constexpr int kWarps = PA_MMA_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 16;  // tokens per tile (the mma M dimension)
constexpr float kLazyLog2 = 8.f;  // the running max moves when a score passes it by 2^8

template <typename T> struct MmaT;
template <> struct MmaT<__nv_bfloat16> {
  __device__ __forceinline__ static void mma(float *d, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <> struct MmaT<__half> {
  __device__ __forceinline__ static void mma(float *d, const uint32_t *a, const uint32_t *b) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

__device__ __forceinline__ void ldsm_x4(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
  return y;
}

// Compile-time shape of one instantiation.
template <int D, int NT>
struct Shape {
  static constexpr int kSteps = D / 16;               // k-steps of S^T, m-tiles of O^T
  static constexpr int kChunks = D / 8;               // 16-byte chunks in a row
  static constexpr int kPitchChunks = (kChunks + 7) / 8 * 8;
  static constexpr int kPitch = kPitchChunks * 16;    // bytes per smem row
  static constexpr int kTileBytes = kTile * kPitch;   // one K (or V) tile
  static constexpr int kStages = D <= 64 ? PA_MMA_STAGES_D64 : D <= 128 ? PA_MMA_STAGES_D128 : 2;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K then V
  static constexpr int kWarpBytes = kStages * kStageBytes;
  static constexpr int kHeads = 8 * NT;               // padded group size
  static constexpr int kRingBytes = kWarps * kWarpBytes;
  static constexpr int kCombineBytes = kWarps * kHeads * (D + 2) * 4;
  static constexpr int kSmemBytes = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
};

// byte offset of (row, chunk) inside a tile: chunks XOR-swizzled by row
template <int D, int NT>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  return row * Shape<D, NT>::kPitch + ((chunk ^ (row & 7)) << 4);
}

// CHUNK: the columns are (query, head) pairs of a chunk (see DecodeParams),
// each with its own causal limit; otherwise they are the group's heads.
template <typename T, int D, int NT, bool MULTI, bool ITEMS, bool CHUNK>
__global__ void __launch_bounds__(kThreads)
    decode_mma_kernel(const DecodeParams p) {
  using S = Shape<D, NT>;
  using M = MmaT<T>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ unsigned s_bad;  // bit s: split s of this CTA met a bad page

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int r = lane >> 2;  // fragment row group
  const int c = lane & 3;   // fragment column pair

  const int hkv = p.num_kv_heads;
  const int g = blockIdx.x % hkv;
  const int G = p.group;  // columns: the group's heads, or a chunk's (query, head) pairs
  // row of column h in q / out (and, times the split count, in the partials)
  auto col_row = [&](int bb, int h) -> size_t {
    if constexpr (CHUNK) {
      const int hg = p.head_group;
      const int i = h / hg;
      return (static_cast<size_t>(bb) * p.chunk_len + i) * p.num_q_heads +
             static_cast<size_t>(g) * hg + (h - i * hg);
    } else {
      return static_cast<size_t>(bb) * p.num_q_heads + static_cast<size_t>(g) * G + h;
    }
  };
  const int bs_log2 = p.block_size_log2;
  const int bs_mask = (1 << bs_log2) - 1;
  const long long cap = static_cast<long long>(p.max_blocks) << bs_log2;

  if (tid == 0) s_bad = 0u;
  pdl_wait();

  // What this CTA reads: split s0 (and the next nsplit - 1) of sequence b,
  // tokens [lo, lo + nsplit * span); in the work-list read, one item.
  int b, s0, nsplit;
  long long lo, span;
  if constexpr (ITEMS) {
    const int4 it = __ldg(reinterpret_cast<const int4 *>(p.items) + blockIdx.x / hkv);
    const int slot = it.w & 0xffff, count = it.w >> 16;
    if (it.x < 0 || it.x >= p.num_seqs || it.y < 0 || it.z < it.y || slot >= count ||
        count > p.num_splits) {
      if (tid == 0) report_error(p.dev_err, PA_DEV_BAD_ITEM);
      return;  // the whole CTA: nothing it could write is known to be its own
    }
    b = it.x;
    s0 = slot;
    nsplit = 1;
    lo = it.y;
    span = static_cast<long long>(it.z) - it.y;
    if (slot == count - 1) {
      // the sequence's last item marks its unused slots empty
      for (int idx = tid; idx < G * (p.num_splits - count); idx += kThreads) {
        const int h = idx / (p.num_splits - count);
        const int s = count + idx - h * (p.num_splits - count);
        const size_t qh = static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G + h;
        p.partial_lse[qh * p.num_splits + s] = -CUDART_INF_F;
      }
    }
  } else {
    b = blockIdx.y;
    s0 = (blockIdx.x / hkv) * p.splits_per_cta;  // first split of this CTA
    nsplit = min(p.splits_per_cta, p.num_splits - s0);
    span = p.pages_per_split > 0 ? static_cast<long long>(p.pages_per_split) << bs_log2 : cap;
    lo = p.pages_per_split > 0 ? static_cast<long long>(s0) * span : 0;
  }

  // The prologue issues its independent loads together: the length, q, and
  // the page ids of this warp's first tiles (read speculatively from the
  // split's first position, index clamped inside the row, validated below).
  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  int pid_pre[S::kStages];
#pragma unroll
  for (int s = 0; s < S::kStages; ++s) {
    const long long pos = lo + (warp + s * kWarps) * kTile + (lane & (kTile - 1));
    pid_pre[s] = __ldg(bt_row + ((pos < cap ? (pos > 0 ? pos : 0) : cap - 1) >> bs_log2));
  }
  int len = __ldg(p.seq_lens + b);

  // ---- Q^T as mma B fragments: lane holds head r, dims 2c,2c+1 (+8) ------
  uint32_t qb[NT][S::kSteps][2];
  {
    const T *qrow = static_cast<const T *>(p.q) +
                    (static_cast<size_t>(b) * p.num_q_heads + static_cast<size_t>(g) * G) * D;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h = nt * 8 + r;
      // a chunk's column h sits in its own query's row
      const T *hrow = CHUNK ? static_cast<const T *>(p.q) + col_row(b, h < G ? h : 0) * D
                            : qrow + h * D;
#pragma unroll
      for (int ks = 0; ks < S::kSteps; ++ks) {
        if (h < G) {
          const T *src = hrow + ks * 16 + 2 * c;
          qb[nt][ks][0] = __ldg(reinterpret_cast<const uint32_t *>(src));
          qb[nt][ks][1] = __ldg(reinterpret_cast<const uint32_t *>(src + 8));
        } else {
          qb[nt][ks][0] = 0u;
          qb[nt][ks][1] = 0u;
        }
      }
    }
  }

  // ---- token range of this CTA -------------------------------------------
  const bool bad_len = (len < 0) || (static_cast<long long>(len) > cap);
  if (bad_len) {
    if (tid == 0) report_error(p.dev_err, PA_DEV_BAD_SEQ_LEN);
    len = 0;
  }
  const int t_begin = static_cast<int>(min(static_cast<long long>(len), lo));
  const int t_end = static_cast<int>(min(static_cast<long long>(len), lo + nsplit * span));
  // CHUNK: last key of this lane's columns 2c, 2c+1 of every n-tile (query i
  // of the chunk sits at len - chunk_len + i)
  int lim[NT][2];
  if constexpr (CHUNK) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        lim[nt][e] = len - p.chunk_len + (nt * 8 + 2 * c + e) / p.head_group;
  }
  // tiles per split (a CTA covers several splits only when a split is whole tiles)
  const int tiles_per_split = MULTI ? static_cast<int>(span / kTile) : 0x7fffffff;

  const T *kpool = static_cast<const T *>(p.k_pool);
  const T *vpool = static_cast<const T *>(p.v_pool);
  unsigned char *ring = smem + warp * S::kWarpBytes;
  const uint32_t ring_u32 = smem_u32(ring);
  __syncthreads();  // s_bad initialised

  const int ntok = t_end - t_begin;
  const int ntiles = ntok > 0 ? (ntok + kTile - 1) / kTile : 0;
  // this warp's tiles: warp, warp + kWarps, ...
  const int my_tiles = ntiles > warp ? (ntiles - warp + kWarps - 1) / kWarps : 0;

  // Page id of token (lane & 15) of this warp's i-th tile (-1 past the end).
  // Fetched one tile ahead of its copies, so the block-table load never sits
  // between a wait and the next copy issue.
  auto fetch_pid = [&](int i) -> int {
    const int pos = t_begin + (warp + i * kWarps) * kTile + (lane & (kTile - 1));
    return (i < my_tiles && pos < t_end) ? __ldg(bt_row + (pos >> bs_log2)) : -1;
  };

  // issue the copies of this warp's i-th tile into stage `stage`; lane j of
  // the first 16 holds the page id of token j of the tile in `pid`
  auto load_tile = [&](int i, int stage, int pid) {
    const int tok0 = t_begin + (warp + i * kWarps) * kTile;
    unsigned char *ks = ring + stage * S::kStageBytes;
    unsigned char *vs = ks + S::kTileBytes;
#pragma unroll
    for (int q = lane; q < kTile * S::kChunks; q += 32) {
      const int row = q / S::kChunks;
      const int chunk = q - row * S::kChunks;
      const int pos = tok0 + row;
      const int page = __shfl_sync(0xffffffffu, pid, row);
      bool valid = pos < t_end;
      const T *ksrc = kpool;
      const T *vsrc = vpool;
      if (valid) {
        if (page < 0 || page >= p.num_pages) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          // the tile lies inside one split: (its index in the CTA) / tiles per split
          atomicOr(&s_bad, MULTI ? 1u << ((warp + i * kWarps) / tiles_per_split) : 1u);
          valid = false;
        } else {
          const size_t prow = (static_cast<size_t>(page) << bs_log2) + (pos & bs_mask);
          const size_t off = (prow * hkv + g) * D + chunk * 8;
          ksrc += off;
          vsrc += off;
        }
      }
      const uint32_t o = tile_off<D, NT>(row, chunk);
      cp_async16(ks + o, ksrc, valid);
      cp_async16(vs + o, vsrc, valid);
    }
  };

#pragma unroll
  for (int s = 0; s < S::kStages - 1; ++s) {
    if (s < my_tiles) load_tile(s, s, pid_pre[s]);
    cp_async_commit();
  }
  int pid_next = pid_pre[S::kStages - 1];

  // running state: heads 2c, 2c+1 of every n-tile
  float m[NT][2], l[NT][2];
  float o[S::kSteps][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt][0] = m[nt][1] = -CUDART_INF_F;
    l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < S::kSteps; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
  }
  const float sl2 = p.scale_log2;

  // Several splits per CTA: combine the warps' states of relative split
  // `srel` and write its partial and lse.  Every warp calls this once per
  // split of the CTA, in order, so the barriers inside always match.
  const int ch = p.comb_heads;
  auto finalize = [&](int srel) {
    // per-lane partial sums of l cover tokens r, r+8 only: finish them
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
        l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
      }
    // the combine area lies past the ring, which keeps filling meanwhile
    float *sm_m = reinterpret_cast<float *>(smem + S::kRingBytes);
    float *sm_l = sm_m + kWarps * ch;  // [warp][head]
    float *sm_o = sm_l + kWarps * ch;  // [warp][head][D]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * c;
      if (h0 < ch) {
        if (r == 0) {
          sm_m[warp * ch + h0] = m[nt][0];
          sm_m[warp * ch + h0 + 1] = m[nt][1];
          sm_l[warp * ch + h0] = l[nt][0];
          sm_l[warp * ch + h0 + 1] = l[nt][1];
        }
#pragma unroll
        for (int mt = 0; mt < S::kSteps; ++mt) {
          const int d0 = mt * 16 + r;
          float *ob = sm_o + (warp * ch + h0) * D;
          ob[d0] = o[mt][nt][0];
          ob[D + d0] = o[mt][nt][1];
          ob[d0 + 8] = o[mt][nt][2];
          ob[D + d0 + 8] = o[mt][nt][3];
        }
      }
    }
    __syncthreads();
    const bool bad = bad_len || ((s_bad >> srel) & 1u);
    const bool is_split = p.pages_per_split > 0;
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int h = idx / D;
      const int d = idx - h * D;
      float Mx = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, sm_m[w * ch + h]);
      float L = 0.f, O = 0.f;
      if (Mx != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float wgt = exp2f(sm_m[w * ch + h] - Mx);
          L = fmaf(sm_l[w * ch + h], wgt, L);
          O = fmaf(sm_o[(w * ch + h) * D + d], wgt, O);
        }
      }
      const bool empty = bad || (Mx == -CUDART_INF_F);
      const float res = empty ? 0.f : O / L;
      const size_t qh = col_row(b, h);
      if (is_split) {
        const size_t row = qh * p.num_splits + s0 + srel;
        p.partial_out[row * D + d] = res;
        if (d == 0)
          p.partial_lse[row] = empty ? -CUDART_INF_F : (Mx + log2f(L)) * 0.69314718055994531f;
      } else {
        static_cast<T *>(p.out)[qh * D + d] = cvt_out<T>(res);
      }
    }
    __syncthreads();  // the combine area is free for the next split
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -CUDART_INF_F;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int mt = 0; mt < S::kSteps; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
    }
  };

  int cur = 0;  // relative split the warp is accumulating
  for (int i = 0; i < my_tiles; ++i) {
    if constexpr (MULTI) {
      while (cur < (warp + i * kWarps) / tiles_per_split) finalize(cur++);
    }
    // Tile i + kStages - 1 goes into the stage tile i - 1 left.  A 2-stage
    // ring refills before waiting for tile i (two tiles in flight during the
    // wait, not one); a 3-stage ring waits first, which measured faster.
    if constexpr (S::kStages > 2) {
      cp_async_wait<S::kStages - 2>();
      __syncwarp();
    } else {
      __syncwarp();  // the reads of tile i - 1's stage are done
    }
    {
      const int ni = i + S::kStages - 1;
      if (ni < my_tiles) {
        load_tile(ni, ni % S::kStages, pid_next);
        pid_next = fetch_pid(ni + 1);
      }
      cp_async_commit();
    }
    if constexpr (S::kStages <= 2) {
      cp_async_wait<S::kStages - 1>();
      __syncwarp();
    }
    const int stage = i % S::kStages;
    const uint32_t ks_u32 = ring_u32 + stage * S::kStageBytes;
    const uint32_t vs_u32 = ks_u32 + S::kTileBytes;
    const int tok0 = t_begin + (warp + i * kWarps) * kTile;

    // S^T = K . Q^T  (rows: tokens r, r+8; columns: heads 2c, 2c+1)
    float sc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
#pragma unroll
    for (int ks = 0; ks < S::kSteps; ++ks) {
      // matrices: (tok 0-7, d lo), (tok 8-15, d lo), (tok 0-7, d hi), (tok 8-15, d hi)
      const int mi = lane >> 3;
      const int row = ((mi & 1) << 3) + (lane & 7);
      const int chunk = ks * 2 + (mi >> 1);
      uint32_t a[4];
      ldsm_x4(a, ks_u32 + tile_off<D, NT>(row, chunk));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) M::mma(sc[nt], a, qb[nt][ks]);
    }

    // online softmax over this tile, per head column
    const bool v0 = tok0 + r < t_end;
    const bool v1 = tok0 + r + 8 < t_end;
    uint32_t pb[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      bool u0 = v0, u1 = v0, u2 = v1, u3 = v1;
      if constexpr (CHUNK) {  // and not past the column's query
        u0 = u0 && tok0 + r <= lim[nt][0];
        u1 = u1 && tok0 + r <= lim[nt][1];
        u2 = u2 && tok0 + r + 8 <= lim[nt][0];
        u3 = u3 && tok0 + r + 8 <= lim[nt][1];
      }
      float s0 = u0 ? sc[nt][0] * sl2 : -CUDART_INF_F;  // token r,   head 2c
      float s1 = u1 ? sc[nt][1] * sl2 : -CUDART_INF_F;  // token r,   head 2c+1
      float s2 = u2 ? sc[nt][2] * sl2 : -CUDART_INF_F;  // token r+8, head 2c
      float s3 = u3 ? sc[nt][3] * sl2 : -CUDART_INF_F;  // token r+8, head 2c+1
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
      // m is a reference max shared by O and l.  It moves only when a lane's
      // score passes it by more than 2^kLazyLog2 (one vote, not a shuffle
      // reduction and a rescale of O on every tile); between moves the
      // exponents below stay under 2^kLazyLog2, and O / l is unchanged.
      if (__any_sync(0xffffffffu, mx0 > m[nt][0] + kLazyLog2 || mx1 > m[nt][1] + kLazyLog2)) {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[nt][0], mx0), mn1 = fmaxf(m[nt][1], mx1);
        // nothing accumulated yet under an infinite reference: O and l are 0
        const float a0 = m[nt][0] == -CUDART_INF_F ? 0.f : ex2_approx(m[nt][0] - mn0);
        const float a1 = m[nt][1] == -CUDART_INF_F ? 0.f : ex2_approx(m[nt][1] - mn1);
        m[nt][0] = mn0;
        m[nt][1] = mn1;
        l[nt][0] *= a0;
        l[nt][1] *= a1;
#pragma unroll
        for (int mt = 0; mt < S::kSteps; ++mt) {
          o[mt][nt][0] *= a0;
          o[mt][nt][1] *= a1;
          o[mt][nt][2] *= a0;
          o[mt][nt][3] *= a1;
        }
      }
      const float mu0 = m[nt][0] == -CUDART_INF_F ? 0.f : m[nt][0];
      const float mu1 = m[nt][1] == -CUDART_INF_F ? 0.f : m[nt][1];
      const float p0 = ex2_approx(s0 - mu0), p1 = ex2_approx(s1 - mu1);  // masked: 2^-inf = 0
      const float p2 = ex2_approx(s2 - mu0), p3 = ex2_approx(s3 - mu1);
      l[nt][0] += p0 + p2;
      l[nt][1] += p1 + p3;
      // P^T blocks (tokens 0-7 | 8-15) x heads, transposed into B fragments
      pb[nt][0] = movmatrix_trans(M::pack(p0, p1));
      pb[nt][1] = movmatrix_trans(M::pack(p2, p3));
    }

    // O^T += V^T . P^T
#pragma unroll
    for (int mt = 0; mt < S::kSteps; ++mt) {
      // matrices of V^T: (d lo, tok 0-7), (d hi, tok 0-7), (d lo, tok 8-15), (d hi, tok 8-15)
      const int mi = lane >> 3;
      const int row = ((mi >> 1) << 3) + (lane & 7);
      const int chunk = mt * 2 + (mi & 1);
      uint32_t a[4];
      ldsm_x4_trans(a, vs_u32 + tile_off<D, NT>(row, chunk));
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) M::mma(o[mt][nt], a, pb[nt]);
    }
  }
  cp_async_wait_all();
  pdl_trigger();  // the merge (or the next read) may start launching
  if constexpr (MULTI) {
    while (cur < nsplit) finalize(cur++);
  } else {
    // One split per CTA: combine once, reusing the ring.
    // per-lane partial sums of l cover tokens r, r+8 only: finish them
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[nt][0] += __shfl_xor_sync(0xffffffffu, l[nt][0], off);
        l[nt][1] += __shfl_xor_sync(0xffffffffu, l[nt][1], off);
      }
    __syncthreads();  // every warp done with its ring: reuse smem for the combine

    float *sm_m = reinterpret_cast<float *>(smem);  // [warp][head]
    float *sm_l = sm_m + kWarps * S::kHeads;         // [warp][head]
    float *sm_o = sm_l + kWarps * S::kHeads;         // [warp][head][D]
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * c;
      if (r == 0) {
        sm_m[warp * S::kHeads + h0] = m[nt][0];
        sm_m[warp * S::kHeads + h0 + 1] = m[nt][1];
        sm_l[warp * S::kHeads + h0] = l[nt][0];
        sm_l[warp * S::kHeads + h0 + 1] = l[nt][1];
      }
#pragma unroll
      for (int mt = 0; mt < S::kSteps; ++mt) {
        const int d0 = mt * 16 + r;
        float *ob = sm_o + (warp * S::kHeads + h0) * D;
        ob[d0] = o[mt][nt][0];
        ob[D + d0] = o[mt][nt][1];
        ob[d0 + 8] = o[mt][nt][2];
        ob[D + d0 + 8] = o[mt][nt][3];
      }
    }
    __syncthreads();

    const bool bad = bad_len || (s_bad != 0u);
    const bool is_split = ITEMS || p.pages_per_split > 0;
    for (int idx = tid; idx < G * D; idx += kThreads) {
      const int h = idx / D;
      const int d = idx - h * D;
      float Mx = -CUDART_INF_F;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) Mx = fmaxf(Mx, sm_m[w * S::kHeads + h]);
      float L = 0.f, O = 0.f;
      if (Mx != -CUDART_INF_F) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float wgt = exp2f(sm_m[w * S::kHeads + h] - Mx);
          L = fmaf(sm_l[w * S::kHeads + h], wgt, L);
          O = fmaf(sm_o[(w * S::kHeads + h) * D + d], wgt, O);
        }
      }
      const bool empty = bad || (Mx == -CUDART_INF_F);
      const float res = empty ? 0.f : O / L;
      const size_t qh = col_row(b, h);
      if (is_split) {
        const size_t row = qh * p.num_splits + s0;
        p.partial_out[row * D + d] = res;
        if (d == 0)
          p.partial_lse[row] = empty ? -CUDART_INF_F : (Mx + log2f(L)) * 0.69314718055994531f;
      } else {
        static_cast<T *>(p.out)[qh * D + d] = cvt_out<T>(res);
      }
    }
  }
}

template <typename T, int D, int NT, bool CHUNK>
cudaError_t launch_shape(DecodeParams p, cudaStream_t stream) {
  using S = Shape<D, NT>;
  auto kern = decode_mma_kernel<T, D, NT, false, false, CHUNK>;
  auto kern_multi = decode_mma_kernel<T, D, NT, true, false, CHUNK>;
  p.splits_per_cta = 1;
  p.comb_heads = S::kHeads;
  int smem = S::kSmemBytes;
  if (p.pages_per_split > 0 && ((p.pages_per_split << p.block_size_log2) % kTile) == 0) {
    // Several splits per CTA when one wave cannot hold a CTA per split but
    // can hold one per (sequence, kv head): the fewest splits per CTA that
    // make the grid fit the resident slots.
    const int ch = p.group <= 4 ? 4 : S::kHeads;
    const int smem_multi = S::kRingBytes + kWarps * ch * (D + 2) * 4;
    int sms = 0, per_sm = 0;
    cudaError_t err = sm_count(&sms);
    if (err == cudaSuccess)
      err = blocks_per_sm(&per_sm, reinterpret_cast<const void *>(kern_multi), kThreads,
                          smem_multi);
    if (err != cudaSuccess) return err;
    const long long pairs = static_cast<long long>(p.num_seqs) * p.num_kv_heads;
    const long long slots = static_cast<long long>(sms) * per_sm;
    if (pairs * p.num_splits > slots && pairs <= slots) {
      const long long groups = slots / pairs;  // CTAs per (sequence, kv head)
      const int k = static_cast<int>((p.num_splits + groups - 1) / groups);
      if (k > 1 && k <= 32) {
        p.splits_per_cta = k;
        p.comb_heads = ch;
        smem = smem_multi;
      }
    }
  }
  const int groups = (p.num_splits + p.splits_per_cta - 1) / p.splits_per_cta;
  dim3 grid(groups * p.num_kv_heads, p.num_seqs);
  if (p.splits_per_cta > 1) return launch_pdl(kern_multi, grid, dim3(kThreads), smem, stream, p);
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, p);
}

template <typename T, int D, int NT>
cudaError_t launch_items_shape(const DecodeParams &p, cudaStream_t stream) {
  using S = Shape<D, NT>;
  auto kern = decode_mma_kernel<T, D, NT, false, true, false>;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), S::kSmemBytes);
  if (err != cudaSuccess) return err;
  dim3 grid(p.num_items * p.num_kv_heads, 1);
  return launch_pdl(kern, grid, dim3(kThreads), S::kSmemBytes, stream, p);
}

template <typename T, int D>
cudaError_t launch_d(const DecodeParams &p, cudaStream_t stream) {
  if (p.items != nullptr) {
    if (p.group <= 8) return launch_items_shape<T, D, 1>(p, stream);
    return launch_items_shape<T, D, 2>(p, stream);
  }
  if (p.chunk_len > 1) {
    if constexpr (D == 64 || D == 128) {
      if (p.group <= 8) return launch_shape<T, D, 1, true>(p, stream);
      if constexpr (D == 64) return launch_shape<T, D, 2, true>(p, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (p.group <= 8) return launch_shape<T, D, 1, false>(p, stream);
  return launch_shape<T, D, 2, false>(p, stream);
}

template <typename T>
cudaError_t launch_typed(const DecodeParams &p, cudaStream_t stream) {
  switch (p.head_dim) {
    case 32: return launch_d<T, 32>(p, stream);
    case 48: return launch_d<T, 48>(p, stream);
    case 64: return launch_d<T, 64>(p, stream);
    case 96: return launch_d<T, 96>(p, stream);
    case 128: return launch_d<T, 128>(p, stream);
    case 256: return launch_d<T, 256>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// Up to 16 columns at head_dim 64 and 8 at head_dim 128: with 16 columns at
// head_dim 128 (two n-tiles, 160+ registers) the chunk kernel measured faster.
bool mma_chunk_supports(pa_dtype dtype, int head_dim, int columns) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  return (head_dim == 64 && columns <= 16) || (head_dim == 128 && columns <= 8);
}

bool mma_supports(pa_dtype dtype, int head_dim, int group) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  if (group > 16) return false;
  switch (head_dim) {
    case 32: case 48: case 64: case 96: case 128: case 256: return true;
  }
  return false;
}

cudaError_t launch_decode_items(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream) {
  return launch_decode_mma(p, dtype, stream);  // p.items selects the work-list variant
}

cudaError_t launch_decode_mma(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_typed<__nv_bfloat16>(p, stream);
  if (dtype == PA_F16) return launch_typed<__half>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
