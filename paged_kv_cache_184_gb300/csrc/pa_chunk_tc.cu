// Chunked multi-query / prefill read on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory).
//
// Same contract as the mma.sync chunk read (nanoserve "Day 23: the real
// triton.jit paged-attention kernel": query i of a chunk sits at position
// past + i and sees tokens 0 .. past + i), for chunks of 128 to 255 (query,
// head) rows per kv head at head_dim 128; longer ones (a prompt's prefill
// among them) go to the warp-specialized read, and at head_dim 64 the
// pipelined one-tile read takes this range.  One CTA owns 128 rows of one
// (sequence, kv head), one row per thread, and walks the causal key range in
// 64-token tiles:
//
//   S [128 x 64] = Q [128 x D] . K_tile^T      tcgen05.mma -> tensor memory
//   softmax      : thread r loads row r of S (tcgen05.ld), masks, takes the
//                  running max and sum in fp32, and writes row r of P
//                  (bf16/f16 pairs) back over the first 32 columns of S
//   O [128 x D] += P . V_tile                 tcgen05.mma with A (P) read from
//                                             tensor memory; O stays there too
//
// P never touches shared memory, which then holds only Q and two K/V stages:
// 97 KB at head_dim 128, two CTAs per SM (256 tensor-memory columns each).
//
// The running max used for the exponent is only moved when a row's max
// grows by more than 2^8 (then O and l are rescaled, warp by warp, through
// tcgen05.ld/st); otherwise P values up to 2^8 are used as they are.  O and
// l always share the same reference max, so the result is the same softmax.
//
// K/V tiles come through the block table ("Three Attention Kernels",
// section "3. Paged KV-cache attention") with 16-byte cp.async copies into
// the swizzled layouts the tensor core reads (K: K-major, V: MN-major), two
// tiles in flight.  Thread 0 issues the MMAs; completion is signalled on an
// mbarrier by tcgen05.commit, and every wait on it is bounded: on time-out
// the kernel records PA_DEV_TIMEOUT, waits (bounded) no further, frees its
// tensor memory and leaves.
//
// In the split read (partial_out set) blockIdx.z picks one fixed page run of
// the sequence ("Three Attention Kernels", section "2. Split-KV
// flash-decoding"); every row stops at the earlier of its causal limit and
// the end of the run, and writes its fp32 partial output and log-sum-exp
// for pa_merge.
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kRows = 128;      // rows per CTA (the MMA M), one per thread
constexpr int kThreads = 128;
constexpr int kKeyTile = 64;    // tokens per tile (the QK MMA N, the PV MMA K)
constexpr float kRescaleLog2 = 8.f;  // move the reference max when it grows by more than 2^8

template <int D>
struct TcShape {
  static constexpr int kQBytes = kRows * D * 2;         // Q: [kb][128 rows][128 B]
  static constexpr int kKVBytes = kKeyTile * D * 2;     // one K or V tile: [kb][64 rows][128 B]
  static constexpr int kSmem = kQBytes + 4 * kKVBytes + 1024;
  static constexpr int kTmemCols = (kKeyTile + D) <= 128 ? 128 : 256;  // S (P over it), then O
  static constexpr int kMinBlocks = D <= 64 ? 4 : 2;                  // CTAs per SM
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, TcShape<D>::kMinBlocks)
    chunk_tc_kernel(const ChunkParams p) {
  using S = TcShape<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t mbar_s, mbar_o;
  __shared__ uint32_t tmem_base;
  __shared__ int s_bad, s_fail;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int hkv = p.num_kv_heads, G = p.group, nq = p.chunk_len;
  const int g = blockIdx.x % hkv;
  const int rows_total = nq * G;
  const int nblk = (rows_total + kRows - 1) / kRows;
  const int rblk = nblk - 1 - blockIdx.x / hkv;  // the longest causal ranges start first
  const int b = blockIdx.y;
  const int split = blockIdx.z;
  const bool partial = p.partial_out != nullptr;
  const int bs_log2 = p.block_size_log2, bs_mask = (1 << bs_log2) - 1;

  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char *sq = smem;                     // Q
  unsigned char *skv = smem + S::kQBytes;       // K0, V0, K1, V1

  if (tid == 0) {
    s_bad = 0;
    s_fail = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar_s)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar_o)));
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&tmem_base)),
                 "n"(S::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  pdl_wait();

  int len = __ldg(p.seq_lens + b);
  const long long cap = static_cast<long long>(p.max_blocks) << bs_log2;
  const bool bad_len = (len < 0) || (static_cast<long long>(len) > cap);
  if (bad_len) {
    if (threadIdx.x == 0) report_error(p.dev_err, PA_DEV_BAD_SEQ_LEN);
    len = 0;
  }
  const int past = len - nq;
  // tokens [t_lo, t_hi) of this CTA: the whole sequence, or one split of it
  int t_lo = 0, t_hi = len;
  if (partial) {
    const long long span = static_cast<long long>(p.pages_per_split) << bs_log2;
    t_lo = static_cast<int>(min(static_cast<long long>(len), split * span));
    t_hi = static_cast<int>(min(static_cast<long long>(len), (split + 1) * span));
  }
  const int row = rblk * kRows + tid;  // this thread's row
  const bool row_ok = row < rows_total;
  const int pos = min(past + row / G, t_hi - 1);  // its last key (inclusive)
  const int last_row = min(rows_total - 1, rblk * kRows + kRows - 1);
  const int kv_end = max(t_lo, min(t_hi, past + last_row / G + 1));
  const int ntiles = (kv_end - t_lo + kKeyTile - 1) / kKeyTile;
  // a warp whose 32 rows are all past the chunk's last row skips the softmax
  // (its rows of O are never stored)
  const bool warp_live = rblk * kRows + warp * 32 < rows_total;

  // ---- Q rows into the swizzled K-major layout ----------------------------
  const T *qbase = static_cast<const T *>(p.q);
  for (int idx = tid; idx < kRows * (D / 8); idx += kThreads) {
    const int r = idx / (D / 8), c = idx - r * (D / 8);
    const int qr = rblk * kRows + r;
    const bool ok = qr < rows_total;
    const T *src = qbase;
    if (ok) {
      const int i = qr / G, h = qr - (qr / G) * G;
      src = qbase + ((static_cast<size_t>(b) * nq + i) * p.num_q_heads +
                     static_cast<size_t>(g) * G + h) * D + c * 8;
    }
    cp_async16(sq + sw_off(r, c, kRows), src, ok);
  }
  cp_async_commit();

  const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
  const T *kpool = static_cast<const T *>(p.k_pool);
  const T *vpool = static_cast<const T *>(p.v_pool);
  // Thread tid copies chunk tid % (D / 8) of rows tid / (D / 8) + k * kRowStep of a tile.
  // Their page ids are read one tile ahead of the copies, so no copy waits for a
  // block-table load.
  constexpr int kCopies = kKeyTile * (D / 8) / kThreads;  // rows per thread: 4, or 8 at 128
  constexpr int kRowStep = kThreads / (D / 8);
  const int c_own = tid % (D / 8), tr0 = tid / (D / 8);
  auto fetch_pages = [&](int j, int (&pid)[kCopies]) {
#pragma unroll
    for (int k = 0; k < kCopies; ++k) {
      const int t = t_lo + j * kKeyTile + tr0 + k * kRowStep;
      pid[k] = (j < ntiles && t < kv_end) ? __ldg(bt_row + (t >> bs_log2)) : -1;
    }
  };
  auto load_tile = [&](int j, int stage, const int (&pid)[kCopies]) {
    unsigned char *ks = skv + (2 * stage) * S::kKVBytes;
    unsigned char *vs = ks + S::kKVBytes;
#pragma unroll
    for (int k = 0; k < kCopies; ++k) {
      const int tr = tr0 + k * kRowStep, c = c_own;
      const int t = t_lo + j * kKeyTile + tr;
      bool valid = t < kv_end;
      const T *ksrc = kpool, *vsrc = vpool;
      if (valid) {
        const int page = pid[k];
        if (page < 0 || page >= p.num_pages) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          s_bad = 1;
          valid = false;
        } else {
          const size_t off =
              (((static_cast<size_t>(page) << bs_log2) + (t & bs_mask)) * hkv + g) * D + c * 8;
          ksrc += off;
          vsrc += off;
        }
      }
      const uint32_t o = sw_off(tr, c, kKeyTile);
      cp_async16(ks + o, ksrc, valid);
      cp_async16(vs + o, vsrc, valid);
    }
  };
  int pid[kCopies];
  fetch_pages(0, pid);
  if (ntiles > 0) load_tile(0, 0, pid);
  cp_async_commit();
  fetch_pages(1, pid);

  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // barrier init, tensor-memory address, s_bad
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const uint32_t t_lane = static_cast<uint32_t>(warp * 32) << 16;  // this warp's 32 lanes
  const uint32_t t_s = tmem, t_o = tmem + kKeyTile;
  const float sl2 = fmaxf(fabsf(p.scale_log2), 1e-30f);
  const bool neg = p.scale_log2 < 0.f;  // a negative scale negates Q . K^T in the MMA
  const uint32_t id_qk = idesc<T>(kRows, kKeyTile, false, neg);
  const uint32_t id_pv = idesc<T>(kRows, D, true, false);
  float m_ref = -CUDART_INF_F;          // reference max (raw units) of the exponent
  float l = 0.f;
  bool fail = false;

  for (int j = 0; j < ntiles; ++j) {
    const int stage = j & 1;
    if (j + 1 < ntiles) load_tile(j + 1, stage ^ 1, pid);
    cp_async_commit();
    fetch_pages(j + 2, pid);  // in flight while this tile is computed
    cp_async_wait<1>();  // Q and tile j are in shared memory
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
    __syncthreads();
    const uint32_t ks_u = smem_u32(skv + (2 * stage) * S::kKVBytes);
    const uint32_t vs_u = ks_u + S::kKVBytes;

    // S = Q . K^T
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
        mma_f16(t_s, sw128_desc(smem_u32(sq) + kb * (kRows * 128) + kin, 16, 1024),
                sw128_desc(ks_u + kb * (kKeyTile * 128) + kin, 16, 1024), id_qk, ks > 0);
      }
      commit(smem_u32(&mbar_s));
    }
    if (!wait_phase(smem_u32(&mbar_s), j & 1)) fail = true;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    if (warp_live) {
      // row `row` of S: mask, running max, probabilities
      float s[kKeyTile];
      tmem_ld64(t_s + t_lane, s);
      const int tok0 = t_lo + j * kKeyTile;
      if (tok0 + kKeyTile - 1 > pos) {  // the tile crosses this row's causal limit
#pragma unroll
        for (int c = 0; c < kKeyTile; ++c)
          if (tok0 + c > pos) s[c] = -CUDART_INF_F;
      }
      const float mx = row_max64(s);
      float alpha = 1.f;
      if (mx != -CUDART_INF_F &&
          (m_ref == -CUDART_INF_F || (mx - m_ref) * sl2 > kRescaleLog2)) {
        alpha = m_ref == -CUDART_INF_F ? 0.f : ex2_approx((m_ref - mx) * sl2);
        m_ref = mx;
      }
      const float mu = m_ref == -CUDART_INF_F ? 0.f : m_ref * sl2;
      const float sum = row_exp64(s, sl2, mu);  // masked: 2^-inf = 0
      l = fmaf(l, alpha, sum);
      // P row over the first 32 columns of S (this thread's lane; its S values
      // are already in registers): tokens 2c and 2c+1 share column c
      {
        uint32_t w[kKeyTile / 2];
#pragma unroll
        for (int c = 0; c < kKeyTile / 2; ++c) w[c] = Pack2<T>::run(s[2 * c], s[2 * c + 1]);
        tmem_st32u(t_s + t_lane, w);
      }
      // rescale this warp's O rows when any of them moved its reference max
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int cb = 0; cb < D; cb += 32) {
          float o[32];
          tmem_ld32(t_o + t_lane + cb, o);
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= alpha;
          tmem_st32(t_o + t_lane + cb, o);
        }
      }
    }  // warp_live
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");

    // O += P . V (each 16-token step of P is 8 columns of tensor memory)
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kKeyTile / 16; ++kk) {
        mma_f16_ta(t_o, t_s + kk * 8, sw128_desc(vs_u + kk * 2048, kKeyTile * 128, 1024), id_pv,
                   (j > 0 || kk > 0));
      }
      commit(smem_u32(&mbar_o));
    }
    if (!wait_phase(smem_u32(&mbar_o), j & 1)) fail = true;
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (__syncthreads_or(fail)) {
      fail = true;
      break;
    }
  }
  cp_async_wait_all();
  pdl_trigger();

  // ---- epilogue: O / l to the output --------------------------------------
  if (fail && tid == 0) report_error(p.dev_err, PA_DEV_TIMEOUT);
  __syncthreads();
  const bool bad = bad_len || s_bad != 0 || fail;
  const bool have_o = ntiles > 0 && !fail;  // uniform over the CTA
  size_t orow = 0;
  if (row_ok) {
    const int i = row / G, h = row - (row / G) * G;
    orow = (static_cast<size_t>(b) * nq + i) * p.num_q_heads + static_cast<size_t>(g) * G + h;
  }
  const bool empty = bad || l == 0.f || !have_o;
  const float inv = empty ? 0.f : 1.f / l;
  // an empty or bad row stores exact zeros (a skipped tile can leave any bits in O)
  auto scaled = [&](float x) { return empty ? 0.f : x * inv; };
  const size_t prow = orow * p.num_splits + split;  // used in the split read only
  if (partial && row_ok)  // natural-log lse of the row's scores over this split
    p.partial_lse[prow] =
        empty ? -CUDART_INF_F : fmaf(m_ref, sl2, log2f(l)) * 0.69314718055994531f;
#pragma unroll
  for (int cb = 0; cb < D; cb += 32) {
    float o[32];
    if (have_o) {
      tmem_ld32(t_o + t_lane + cb, o);  // all lanes: the load is warp-collective
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = 0.f;
    }
    if (row_ok && partial) {
      float *dst = p.partial_out + prow * D + cb;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4 *>(dst + e) =
            make_float4(scaled(o[e]), scaled(o[e + 1]), scaled(o[e + 2]), scaled(o[e + 3]));
    } else if (row_ok) {
      T *dst = static_cast<T *>(p.out) + orow * D + cb;
#pragma unroll
      for (int e = 0; e < 32; e += 8) {
        uint4 w;
        w.x = Pack2<T>::run(scaled(o[e]), scaled(o[e + 1]));
        w.y = Pack2<T>::run(scaled(o[e + 2]), scaled(o[e + 3]));
        w.z = Pack2<T>::run(scaled(o[e + 4]), scaled(o[e + 5]));
        w.w = Pack2<T>::run(scaled(o[e + 6]), scaled(o[e + 7]));
        *reinterpret_cast<uint4 *>(dst + e) = w;
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 0) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(S::kTmemCols));
  }
}

template <typename T, int D>
cudaError_t launch_d(const ChunkParams &p, cudaStream_t stream) {
  auto kern = chunk_tc_kernel<T, D>;
  const int smem = TcShape<D>::kSmem;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  const int nblk = (p.chunk_len * p.group + kRows - 1) / kRows;
  dim3 grid(nblk * p.num_kv_heads, p.num_seqs, p.partial_out ? p.num_splits : 1);
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, p);
}

template <typename T>
cudaError_t launch_t(const ChunkParams &p, cudaStream_t stream) {
  if (p.head_dim == 128) return launch_d<T, 128>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

// At head_dim 128 this read measured faster than the mma.sync one from a full
// 128-row tile per (sequence, kv head) on.  (At head_dim 64 it was faster from
// 64 rows on, and the pipelined read is faster still: 16-query chunks of the
// 64 x 4096-token batch took 129.2 us here, 112.3 us there.)
bool chunk_tc_supports(pa_dtype dtype, int head_dim, int rows) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  return head_dim == 128 && rows >= kRows;
}

cudaError_t launch_chunk_tc(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_t<__nv_bfloat16>(p, stream);
  if (dtype == PA_F16) return launch_t<__half>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
