// Chunked multi-query paged read on the tensor cores (mma.sync m16n8k16).
//
// nanoserve "Day 23: the real triton.jit paged-attention kernel" gives each
// query position i of a chunk its own program, with a causal offset: query i
// sits at position past + i and attends to tokens 0 .. past + i.  Here a
// sequence's chunk of n_q queries and the G query heads of one kv head form
// n_q * G rows (query-major: row = i * G + h), and the rows are the M side
// of the matrix products:
//
//   S [16 rows x 8 tokens]  = Q_rows [16 x D] . K_tile^T [D x 8]
//   O [16 rows x D]        += P [16 x 16 tokens] . V_tile [16 x D]
//
// One CTA per (sequence, kv head, block of 64 rows); each of its 4 warps owns
// one 16-row m-tile over the CTA's whole causal key range, so no warp needs
// another's state.  The warps share 64-token K/V tiles that the CTA streams
// through a 3-stage cp.async ring (XOR-swizzled rows, page ids read through
// the block table as in "Three Attention Kernels" section "3. Paged KV-cache
// attention").  The online softmax runs per row in fp32; P leaves the S
// accumulators as the A fragments of the second product without touching
// shared memory.  Keys past a row's position are masked to -inf; a query at
// a negative position sees nothing and its output is 0.
//
// The split read ("Three Attention Kernels", section "2. Split-KV
// flash-decoding", applied to the chunk) runs the same CTA over one fixed
// page run of the sequence (blockIdx.z): each row keeps the part of the run
// at or before its causal limit and writes its fp32 partial output and
// log-sum-exp for pa_merge instead of the final row.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRowsPerCta = kWarps * 16;
constexpr int kKeyTile = 64;  // tokens per pipeline stage
constexpr int kStages = 3;

template <typename T> struct Mma;
template <> struct Mma<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};
template <> struct Mma<__half> {
  __device__ __forceinline__ static void run(float *d, const uint32_t *a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
  __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
};

__device__ __forceinline__ void ldsm4(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm4_t(uint32_t *r, uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <int D>
struct ChunkShape {
  static constexpr int kSteps = D / 16;  // k-steps of Q.K^T
  static constexpr int kDTiles = D / 8;  // n-tiles of P.V (even)
  static constexpr int kChunks = D / 8;  // 16-byte chunks per row
  static constexpr int kPitch = (kChunks + 7) / 8 * 8 * 16;
  static constexpr int kTileBytes = kKeyTile * kPitch;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes;
};

template <int D>
__device__ __forceinline__ uint32_t toff(int row, int chunk) {
  return row * ChunkShape<D>::kPitch + ((chunk ^ (row & 7)) << 4);
}

// Up to head_dim 64, 128 registers keep 4 CTAs (512 threads) per SM, which
// measured faster than the unbounded allocation; wider heads need more.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads, D <= 64 ? 4 : 1) chunk_kernel(const ChunkParams p) {
  using S = ChunkShape<D>;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_bad;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, c = lane & 3;
  const int hkv = p.num_kv_heads, G = p.group, nq = p.chunk_len;
  const int g = blockIdx.x % hkv;
  const int rblk = blockIdx.x / hkv;
  const int b = blockIdx.y;
  const int split = blockIdx.z;
  const bool partial = p.partial_out != nullptr;
  const int bs_log2 = p.block_size_log2, bs_mask = (1 << bs_log2) - 1;
  const int rows_total = nq * G;

  if (tid == 0) s_bad = 0;
  pdl_wait();

  int len = __ldg(p.seq_lens + b);
  const long long cap = static_cast<long long>(p.max_blocks) << bs_log2;
  const bool bad_len = (len < 0) || (static_cast<long long>(len) > cap);
  if (bad_len) {
    if (tid == 0) report_error(p.dev_err, PA_DEV_BAD_SEQ_LEN);
    len = 0;
  }
  const int past = len - nq;  // position of query 0 (may be negative)
  // tokens [t_lo, t_hi) of this CTA: the whole sequence, or one split of it
  int t_lo = 0, t_hi = len;
  if (partial) {
    const long long span = static_cast<long long>(p.pages_per_split) << bs_log2;
    t_lo = static_cast<int>(min(static_cast<long long>(len), split * span));
    t_hi = static_cast<int>(min(static_cast<long long>(len), (split + 1) * span));
  }

  // rows of this warp and of this thread's two fragment rows
  const int row0 = rblk * kRowsPerCta + warp * 16;
  const int ra = row0 + r, rb = row0 + r + 8;
  // last key of row ra (inclusive): its causal limit, or the end of the split
  const int pos_a = min(past + ra / G, t_hi - 1);
  const int pos_b = min(past + rb / G, t_hi - 1);
  // key range of the CTA and of the warp
  const int cta_last_row = min(rows_total - 1, rblk * kRowsPerCta + kRowsPerCta - 1);
  const int kv_end = max(t_lo, min(t_hi, past + cta_last_row / G + 1));
  const int warp_last_row = min(rows_total - 1, row0 + 15);
  const int warp_end =
      row0 < rows_total ? max(t_lo, min(t_hi, past + warp_last_row / G + 1)) : t_lo;

  // Q rows as A fragments
  uint32_t qa[S::kSteps][4];
  {
    const T *qb = static_cast<const T *>(p.q);
    auto qptr = [&](int row) -> const T * {
      const int i = row / G, h = row - (row / G) * G;
      return qb + ((static_cast<size_t>(b) * nq + i) * p.num_q_heads +
                   static_cast<size_t>(g) * G + h) * D;
    };
    const bool va = ra < rows_total, vb = rb < rows_total;
    const T *pa_ = va ? qptr(ra) : qb;
    const T *pb_ = vb ? qptr(rb) : qb;
    // a negative scale is applied as a sign flip of q, so the scale that
    // scores meet is never negative (the running max stays a max)
    const uint32_t flip = p.scale_log2 < 0.f ? 0x80008000u : 0u;
#pragma unroll
    for (int ks = 0; ks < S::kSteps; ++ks) {
      const int d0 = ks * 16 + 2 * c;
      qa[ks][0] = va ? __ldg(reinterpret_cast<const uint32_t *>(pa_ + d0)) ^ flip : 0u;
      qa[ks][1] = vb ? __ldg(reinterpret_cast<const uint32_t *>(pb_ + d0)) ^ flip : 0u;
      qa[ks][2] = va ? __ldg(reinterpret_cast<const uint32_t *>(pa_ + d0 + 8)) ^ flip : 0u;
      qa[ks][3] = vb ? __ldg(reinterpret_cast<const uint32_t *>(pb_ + d0 + 8)) ^ flip : 0u;
    }
  }
  // smallest key limit among this warp's rows: tiles ending at or below it need no mask
  const int warp_min_pos = min(past + row0 / G, t_hi - 1);

  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  const T *kpool = static_cast<const T *>(p.k_pool);
  const T *vpool = static_cast<const T *>(p.v_pool);
  const uint32_t ring = smem_u32(smem);
  __syncthreads();  // s_bad initialised

  auto load_tile = [&](int j, int stage) {
    unsigned char *ks = smem + stage * S::kStageBytes;
    unsigned char *vs = ks + S::kTileBytes;
    const int tok0 = t_lo + j * kKeyTile;
#pragma unroll
    for (int q = tid; q < kKeyTile * S::kChunks; q += kThreads) {
      const int row = q / S::kChunks;
      const int chunk = q - row * S::kChunks;
      const int pos = tok0 + row;
      bool valid = pos < kv_end;
      const T *ksrc = kpool, *vsrc = vpool;
      if (valid) {
        const int page = __ldg(bt_row + (pos >> bs_log2));
        if (page < 0 || page >= p.num_pages) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          s_bad = 1;
          valid = false;
        } else {
          const size_t off =
              (((static_cast<size_t>(page) << bs_log2) + (pos & bs_mask)) * hkv + g) * D + chunk * 8;
          ksrc += off;
          vsrc += off;
        }
      }
      const uint32_t o = toff<D>(row, chunk);
      cp_async16(ks + o, ksrc, valid);
      cp_async16(vs + o, vsrc, valid);
    }
  };

  const int ntiles = (kv_end - t_lo + kKeyTile - 1) / kKeyTile;
#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) load_tile(s, s);
    cp_async_commit();
  }

  float o[S::kDTiles][4];
#pragma unroll
  for (int n = 0; n < S::kDTiles; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  float m_a = -CUDART_INF_F, m_b = -CUDART_INF_F, l_a = 0.f, l_b = 0.f;
  // |scale| * log2(e), kept at least 1e-30 so that a masked score (-inf) times it
  // stays -inf when scale is 0; raw scores times 1e-30 are 0 to fp32 precision
  const float sl2 = fmaxf(fabsf(p.scale_log2), 1e-30f);

  for (int j = 0; j < ntiles; ++j) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nj = j + kStages - 1;
      if (nj < ntiles) load_tile(nj, nj % kStages);
      cp_async_commit();
    }
    const int tok0 = t_lo + j * kKeyTile;
    if (tok0 >= warp_end) continue;  // every row of this warp is past its limit
    const uint32_t ks_u = ring + (j % kStages) * S::kStageBytes;
    const uint32_t vs_u = ks_u + S::kTileBytes;

    // S = Q . K^T over 8 n-tiles of 8 tokens
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[n][e] = 0.f;
    const int mi = lane >> 3;
#pragma unroll
    for (int ks = 0; ks < S::kSteps; ++ks) {
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        // (tok n*8.., d lo), (tok n*8.., d hi), (tok (n+1)*8.., d lo), (tok (n+1)*8.., d hi)
        const int row = n * 8 + ((mi >> 1) << 3) + (lane & 7);
        const int chunk = ks * 2 + (mi & 1);
        uint32_t kb[4];
        ldsm4(kb, ks_u + toff<D>(row, chunk));
        Mma<T>::run(sc[n], qa[ks], kb[0], kb[1]);
        Mma<T>::run(sc[n + 1], qa[ks], kb[2], kb[3]);
      }
    }

    // causal mask (only on tiles that cross a row's limit) and the row max,
    // in raw score units; the scale is applied inside the exponent below
    if (tok0 + kKeyTile - 1 > warp_min_pos) {
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int t = tok0 + n * 8 + 2 * c;
        if (t > pos_a) sc[n][0] = -CUDART_INF_F;
        if (t + 1 > pos_a) sc[n][1] = -CUDART_INF_F;
        if (t > pos_b) sc[n][2] = -CUDART_INF_F;
        if (t + 1 > pos_b) sc[n][3] = -CUDART_INF_F;
      }
    }
    float mx_a = -CUDART_INF_F, mx_b = -CUDART_INF_F;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      mx_a = fmaxf(mx_a, fmaxf(sc[n][0], sc[n][1]));
      mx_b = fmaxf(mx_b, fmaxf(sc[n][2], sc[n][3]));
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
      mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, off));
      mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, off));
    }
    const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
    const float mu_a = mn_a == -CUDART_INF_F ? 0.f : mn_a * sl2;  // scaled max
    const float mu_b = mn_b == -CUDART_INF_F ? 0.f : mn_b * sl2;
    const float al_a = m_a == -CUDART_INF_F ? 0.f : ex2_approx(fmaf(m_a, sl2, -mu_a));
    const float al_b = m_b == -CUDART_INF_F ? 0.f : ex2_approx(fmaf(m_b, sl2, -mu_b));
    m_a = mn_a;
    m_b = mn_b;
    float sum_a = 0.f, sum_b = 0.f;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      sc[n][0] = ex2_approx(fmaf(sc[n][0], sl2, -mu_a));  // exp2(-inf) = 0 for masked keys
      sc[n][1] = ex2_approx(fmaf(sc[n][1], sl2, -mu_a));
      sc[n][2] = ex2_approx(fmaf(sc[n][2], sl2, -mu_b));
      sc[n][3] = ex2_approx(fmaf(sc[n][3], sl2, -mu_b));
      sum_a += sc[n][0] + sc[n][1];
      sum_b += sc[n][2] + sc[n][3];
    }
    l_a = fmaf(l_a, al_a, sum_a);
    l_b = fmaf(l_b, al_b, sum_b);
#pragma unroll
    for (int n = 0; n < S::kDTiles; ++n) {
      o[n][0] *= al_a;
      o[n][1] *= al_a;
      o[n][2] *= al_b;
      o[n][3] *= al_b;
    }

    // O += P . V, 16 tokens per k-step
#pragma unroll
    for (int kk = 0; kk < kKeyTile / 16; ++kk) {
      uint32_t pa[4];
      pa[0] = Mma<T>::pack(sc[2 * kk][0], sc[2 * kk][1]);
      pa[1] = Mma<T>::pack(sc[2 * kk][2], sc[2 * kk][3]);
      pa[2] = Mma<T>::pack(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
      pa[3] = Mma<T>::pack(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
#pragma unroll
      for (int dn = 0; dn < S::kDTiles; dn += 2) {
        // (tok 0-7, d dn), (tok 8-15, d dn), (tok 0-7, d dn+1), (tok 8-15, d dn+1)
        const int row = kk * 16 + ((mi & 1) << 3) + (lane & 7);
        const int chunk = dn + (mi >> 1);
        uint32_t vb[4];
        ldsm4_t(vb, vs_u + toff<D>(row, chunk));
        Mma<T>::run(o[dn], pa, vb[0], vb[1]);
        Mma<T>::run(o[dn + 1], pa, vb[2], vb[3]);
      }
    }
  }
  cp_async_wait_all();
  pdl_trigger();
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  __syncthreads();  // s_bad final
  const bool bad = bad_len || (s_bad != 0);

  auto store_row = [&](int row, float l, float m, int e0) {
    if (row >= rows_total) return;
    const int i = row / G, h = row - (row / G) * G;
    const size_t orow = (static_cast<size_t>(b) * nq + i) * p.num_q_heads +
                        static_cast<size_t>(g) * G + h;
    const bool empty = bad || l == 0.f;
    const float inv = empty ? 0.f : 1.f / l;
    if (partial) {
      const size_t prow = orow * p.num_splits + split;
      float *dst = p.partial_out + prow * D;
#pragma unroll
      for (int n = 0; n < S::kDTiles; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8 + 2 * c) =
            make_float2(o[n][e0] * inv, o[n][e0 + 1] * inv);
      // natural-log lse of the row's scores over this split
      if (c == 0)
        p.partial_lse[prow] =
            empty ? -CUDART_INF_F : fmaf(m, sl2, log2f(l)) * 0.69314718055994531f;
      return;
    }
    T *dst = static_cast<T *>(p.out) + orow * D;
#pragma unroll
    for (int n = 0; n < S::kDTiles; ++n) {
      const int d = n * 8 + 2 * c;
      dst[d] = cvt_out<T>(o[n][e0] * inv);
      dst[d + 1] = cvt_out<T>(o[n][e0 + 1] * inv);
    }
  };
  store_row(ra, l_a, m_a, 0);
  store_row(rb, l_b, m_b, 2);
}

template <typename T, int D>
cudaError_t launch_d(const ChunkParams &p, cudaStream_t stream) {
  auto kern = chunk_kernel<T, D>;
  const int smem = ChunkShape<D>::kSmemBytes;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  const int rblocks = (p.chunk_len * p.group + kRowsPerCta - 1) / kRowsPerCta;
  dim3 grid(rblocks * p.num_kv_heads, p.num_seqs, p.partial_out ? p.num_splits : 1);
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, p);
}

template <typename T>
cudaError_t launch_t(const ChunkParams &p, cudaStream_t stream) {
  switch (p.head_dim) {
    case 32: return launch_d<T, 32>(p, stream);
    case 48: return launch_d<T, 48>(p, stream);
    case 64: return launch_d<T, 64>(p, stream);
    case 96: return launch_d<T, 96>(p, stream);
    case 128: return launch_d<T, 128>(p, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool chunk_supports(pa_dtype dtype, int head_dim) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  switch (head_dim) {
    case 32: case 48: case 64: case 96: case 128: return true;
  }
  return false;
}

int chunk_rows_per_cta() { return kRowsPerCta; }

cudaError_t launch_chunk(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_t<__nv_bfloat16>(p, stream);
  if (dtype == PA_F16) return launch_t<__half>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
