// Pipelined chunked read on the tcgen05 tensor cores: one 128-row Q tile per
// CTA, the phases of a key tile on different warps, S double-buffered.
//
// Same contract as the other chunk reads (nanoserve "Day 23: the real
// triton.jit paged-attention kernel": query i of a chunk sits at position
// past + i and sees tokens 0 .. past + i) and the same per-row arithmetic as
// the warp-specialized read (fp32 online softmax with a lazily moved
// reference max, P rounded to the cache dtype).  It serves chunks of up to 255
// (query, head) rows per kv head: too few rows for two Q tiles per CTA, so
// several CTAs share an SM and each keeps its own K/V stream going.
//
// Run in order, every key tile costs QK, a tensor-memory round trip, the
// softmax, and P.V with another round trip.  Here the phases overlap:
//
//   warps 0-3   softmax: thread r owns row r (tensor-memory lane r), reads its
//               S row, writes its P row back over S as 16-bit pairs, and moves
//               the reference max (rescaling its O row) only when a score
//               passes it by more than 2^8; warps with no row of the chunk
//               stop at once
//   warp 4      lane 0 issues S(j) = Q . K_j^T into S buffer j % 2 and
//               O += P(j) . V_j, each committed to an mbarrier; QK(j + 2) goes
//               as soon as P.V(j) has finished reading P(j) from that buffer,
//               so S(j + 1) is ready while the softmax works on tile j
//   warp 5      loads KT-token K/V tiles through the block table ("Three
//               Attention Kernels", section "3. Paged KV-cache attention")
//               into a ring: whole tiles by 2D tensor-map copies (one per page
//               and head_dim half, counted in bytes on the stage's `full`
//               mbarrier), a ragged last tile (or pages of fewer than 8
//               tokens) by 16-byte cp.async with zero-fill
//
// Tensor memory: S_0 | S_1 (32 columns each) | O (head_dim columns).  Key
// tiles are 32 tokens so that at head_dim 64 the three take 128 columns and
// four CTAs (49 KB of shared memory each) share an SM; at head_dim 128 they
// take 192 (256 allocated) and two CTAs (97 KB each) share one.  A 128 x 32 x
// 16 product costs the tensor pipe about as long as a 128 x 64 x 16 one (~50
// cycles, measured), so QK takes twice the pipe time per key that 64-token
// tiles would; with four CTAs per SM the pipe still has room.
//
// mbarriers: full/empty per ring stage, and per S buffer s (S ready), p (P
// written, one arrival per live softmax warp) and o (P.V done: buffer and O
// free).  No barrier can complete twice before its waiter looks: each next
// completion needs the waiter's own progress.  Every wait is bounded (about
// a second); on time-out the kernel records PA_DEV_TIMEOUT, every role leaves
// its loop, the outputs are zeroed and the tensor memory is freed.
//
// In the split read (partial_out set) blockIdx.z picks one fixed page run of
// the sequence ("Three Attention Kernels", section "2. Split-KV
// flash-decoding"); each row stops at the earlier of its causal limit and the
// end of the run and writes its fp32 partial output and log-sum-exp.
#include <cuda.h>
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kRows = 128;  // rows of the Q tile (the MMA M), one per softmax thread
constexpr int kSoftmaxWarps = 4;
constexpr int kMmaWarp = 4, kLoadWarp = 5;
constexpr int kThreads = 192;
constexpr float kRescaleLog2 = 8.f;

// Shape per head_dim: key-tile tokens, ring stages, CTAs per SM.
template <int D> struct PipeShape;
template <> struct PipeShape<64> {
  static constexpr int kKeyTile = 32, kStages = 4, kMinBlocks = 4;
};
template <> struct PipeShape<128> {
  static constexpr int kKeyTile = 32, kStages = 4, kMinBlocks = 2;
};

template <int D>
struct PipeSizes : PipeShape<D> {
  using B = PipeShape<D>;
  static constexpr int kQBytes = kRows * D * 2;           // Q: [kb][128 rows][128 B]
  static constexpr int kKVBytes = B::kKeyTile * D * 2;    // K or V tile: [kb][KT rows][128 B]
  static constexpr int kSmem = kQBytes + B::kStages * 2 * kKVBytes + 1024;
  static constexpr int kTmemUsed = 2 * B::kKeyTile + D;   // S_0, S_1, O
  static constexpr int kTmemCols = kTmemUsed <= 128 ? 128 : 256;
  static_assert(kTmemUsed <= 256, "tensor memory");
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, PipeShape<D>::kMinBlocks)
    chunk_tc_pipe_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v, const int use_tma,
                         const int withhold) {
  using S = PipeSizes<D>;
  constexpr int KT = S::kKeyTile;
  constexpr int kStages = S::kStages;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ uint64_t bar_s[2], bar_p[2], bar_o[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_bad, s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = p.num_kv_heads, G = p.group, nq = p.chunk_len;
  const int g = blockIdx.x % hkv;
  const int rows_total = nq * G;
  const int nblk = (rows_total + kRows - 1) / kRows;
  const int rblk = nblk - 1 - blockIdx.x / hkv;  // the longest causal ranges start first
  const int b = blockIdx.y;
  const int split = blockIdx.z;
  const bool partial = p.partial_out != nullptr;
  const int bs_log2 = p.block_size_log2, bs_mask = (1 << bs_log2) - 1;
  const int base0 = rblk * kRows;
  // softmax warps that hold a row of the chunk (at least one: base0 < rows_total)
  const int live_warps = min(kSoftmaxWarps, (rows_total - base0 + 31) / 32);

  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char *sq = smem;                // Q
  unsigned char *skv = smem + S::kQBytes;  // stage st: K at 2*st, V at 2*st + 1

  if (tid == 0) {
    s_bad = 0;
    s_fail = 0;
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], 1);
    }
#pragma unroll
    for (int nb = 0; nb < 2; ++nb) {
      mbar_init(&bar_s[nb], 1);
      mbar_init(&bar_p[nb], live_warps);
      mbar_init(&bar_o[nb], 1);
    }
  }
  if (warp == kMmaWarp) {
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
  const int last_row = min(rows_total - 1, base0 + kRows - 1);
  const int kv_end = max(t_lo, min(t_hi, past + last_row / G + 1));
  const int ntiles = (kv_end - t_lo + KT - 1) / KT;

  // ---- Q rows into the swizzled K-major layout (all threads) --------------
  const T *qbase = static_cast<const T *>(p.q);
  for (int idx = tid; idx < kRows * (D / 8); idx += kThreads) {
    const int r = idx / (D / 8), c = idx - r * (D / 8);
    const int qr = base0 + r;
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
  cp_async_wait_all();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // barriers, tensor-memory address, Q
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  bool fail = false;

  // softmax-thread state (warps 0-3): row base0 + tid, tensor-memory lane tid
  const bool warp_live = warp < live_warps;  // a softmax warp with rows of the chunk
  const int row = base0 + tid;
  const bool row_ok = warp_live && row < rows_total;
  const float sl2 = fmaxf(fabsf(p.scale_log2), 1e-30f);
  float m_ref = -CUDART_INF_F;  // reference max (raw units) of the exponent
  float l = 0.f;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ load warp
    // Tile j goes to stage j % kStages once P.V(j - kStages) has released it.
    // Lane l holds the id of page first + l of its tile (a 32-token tile spans
    // at most 32 pages), read one tile ahead; an id outside the pool is
    // reported, marks the outputs bad and reads as -1 (no copy).
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
    const T *kpool = static_cast<const T *>(p.k_pool);
    const T *vpool = static_cast<const T *>(p.v_pool);
    static_assert(KT == 32, "one page id per lane");
    auto fetch_page = [&](int j) -> int {
      int pa = -1;
      if (j < ntiles) {
        const int t0 = t_lo + j * KT;
        const int first = t0 >> bs_log2;
        const int last = (min(t0 + KT, kv_end) - 1) >> bs_log2;  // < max_blocks
        if (first + lane <= last) {
          pa = __ldg(bt_row + first + lane);
          if (pa < 0 || pa >= p.num_pages) {
            report_error(p.dev_err, PA_DEV_BAD_PAGE);
            s_bad = 1;
            pa = -1;
          }
        }
      }
      return pa;
    };
    // one lane waits, the warp follows its answer (keeps the warp converged)
    auto warp_wait = [&](uint64_t *bar, uint32_t phase) -> bool {
      int ok = 1;
      if (lane == 0) ok = wait_phase(smem_u32(bar), phase) ? 1 : 0;
      return __shfl_sync(0xffffffffu, ok, 0) != 0;
    };
    int pa = fetch_page(0);
    // test hook: no tile is ever announced, so the other roles' waits run out
    for (int j = 0; j < ntiles && !withhold; ++j) {
      const int st = j % kStages;
      if (j >= kStages && !warp_wait(&bar_empty[st], ((j / kStages) - 1) & 1)) {
        fail = true;
        break;
      }
      unsigned char *ks = skv + (2 * st) * S::kKVBytes;
      unsigned char *vs = ks + S::kKVBytes;
      const int t0 = t_lo + j * KT;
      const int first = t0 >> bs_log2;
      const int na = fetch_page(j + 1);
      if (use_tma && t0 + KT <= kv_end) {
        // pages of the tile: KT / bs of them (bs < KT), or one KT-row part of a page
        const int rows = bs_log2 >= 5 ? KT : (1 << bs_log2);
        const int npg = KT / rows;  // <= KT / 8 (bs >= 8)
        int pg[KT / 8];
#pragma unroll
        for (int i = 0; i < KT / 8; ++i) pg[i] = __shfl_sync(0xffffffffu, pa, i);
        if (lane == 0) {
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < KT / 8; ++i)
            if (i < npg && pg[i] >= 0) bytes += 2u * rows * D * 2u;
          mbar_arrive_expect(&bar_full[st], bytes);
#pragma unroll
          for (int i = 0; i < KT / 8; ++i) {
            if (i >= npg || pg[i] < 0) continue;  // a bad page: the outputs are zeroed anyway
            const int y = (pg[i] << bs_log2) + (rows == KT ? (t0 & bs_mask) : 0);
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb) {
              const uint32_t off = kb * (KT * 128) + i * rows * 128;
              tma_load_2d(ks + off, &tmap_k, g * D + kb * 64, y, &bar_full[st]);
              tma_load_2d(vs + off, &tmap_v, g * D + kb * 64, y, &bar_full[st]);
            }
          }
        }
        __syncwarp();
        pa = na;
        continue;
      }
#pragma unroll 4
      for (int idx = lane; idx < KT * (D / 8); idx += 32) {
        const int tr = idx / (D / 8), c = idx % (D / 8);
        const int t = t0 + tr;
        const int pi = (t >> bs_log2) - first;  // 0 .. KT - 1
        const int page = __shfl_sync(0xffffffffu, pa, pi);
        const bool valid = t < kv_end && page >= 0;
        const size_t off =
            valid ? (((static_cast<size_t>(page) << bs_log2) + (t & bs_mask)) * hkv + g) * D + c * 8
                  : 0;
        const uint32_t o = sw_off(tr, c, KT);
        cp_async16(ks + o, kpool + off, valid);
        cp_async16(vs + o, vpool + off, valid);
      }
      cp_async_commit();
      pa = na;
      cp_async_wait_all();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[st]);
    }
    // wait for the last stages' releases, so that no arrival reaches this
    // CTA's shared memory after it exits
    for (int j = max(0, ntiles - kStages); j < ntiles && !fail; ++j)
      if (!warp_wait(&bar_empty[j % kStages], (j / kStages) & 1)) fail = true;
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA warp
    if (lane == 0) {
      const uint32_t id_qk = idesc<T>(kRows, KT, false, p.scale_log2 < 0.f);
      const uint32_t id_pv = idesc<T>(kRows, D, true, false);
      const uint32_t qs_u = smem_u32(sq);
      const uint32_t t_o = tmem + 2 * KT;
      // S(j) = Q . K_j^T into buffer j % 2, once tile j is in and P.V(j - 2)
      // has finished reading that buffer
      auto issue_qk = [&](int j) -> bool {
        if (!wait_phase(smem_u32(&bar_full[j % kStages]), (j / kStages) & 1)) return false;
        if (j >= 2 && !wait_phase(smem_u32(&bar_o[j & 1]), ((j >> 1) - 1) & 1)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t ks_u = smem_u32(skv + (2 * (j % kStages)) * S::kKVBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
          mma_f16(tmem + (j & 1) * KT, sw128_desc(qs_u + kb * (kRows * 128) + kin, 16, 1024),
                  sw128_desc(ks_u + kb * (KT * 128) + kin, 16, 1024), id_qk, ks > 0);
        }
        commit(smem_u32(&bar_s[j & 1]));
        return true;
      };
      // O += P(j) . V_j once every live softmax warp has written its P rows;
      // its completion frees the S buffer, the ring stage and O
      auto issue_pv = [&](int j) -> bool {
        if (!wait_phase(smem_u32(&bar_p[j & 1]), (j >> 1) & 1)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t vs_u = smem_u32(skv + (2 * (j % kStages) + 1) * S::kKVBytes);
        const uint32_t t_s = tmem + (j & 1) * KT;
#pragma unroll
        for (int kk = 0; kk < KT / 16; ++kk)
          mma_f16_ta(t_o, t_s + kk * 8, sw128_desc(vs_u + kk * 2048, KT * 128, 1024), id_pv,
                     (j > 0 || kk > 0));
        commit(smem_u32(&bar_o[j & 1]));
        commit(smem_u32(&bar_empty[j % kStages]));
        return true;
      };
      for (int j = 0; j < 2 && j < ntiles && !fail; ++j)
        if (!issue_qk(j)) fail = true;
      for (int j = 0; j < ntiles && !fail; ++j) {
        if (!issue_pv(j)) {
          fail = true;
          break;
        }
        if (j + 2 < ntiles && !issue_qk(j + 2)) fail = true;
      }
    }
    __syncwarp();
  } else if (warp_live) {
    // --------------------------------------------------------- softmax warps
    const uint32_t t_lane = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_o = tmem + 2 * KT + t_lane;
    const int pos = min(past + row / G, t_hi - 1);  // this row's last key (inclusive)
    for (int j = 0; j < ntiles; ++j) {
      if (!wait_phase(smem_u32(&bar_s[j & 1]), (j >> 1) & 1)) fail = true;
      if (__any_sync(0xffffffffu, fail)) {
        fail = true;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t t_s = tmem + (j & 1) * KT + t_lane;
      const int tok0 = t_lo + j * KT;
      float s[KT];
      // S row of this thread, -inf past its last key (warp-collective load)
      auto load_s = [&]() {
        if constexpr (KT == 32) {
          tmem_ld32(t_s, s);
        } else {
          tmem_ld64(t_s, s);
        }
        if (tok0 + KT - 1 > pos) {  // the tile crosses this row's last key
#pragma unroll
          for (int c = 0; c < KT; ++c)
            if (tok0 + c > pos) s[c] = -CUDART_INF_F;
        }
      };
      load_s();
      // Common case first: exponents against the current reference.  When their
      // sum is at most 2^8 no probability exceeds 2^8, so the lazy rule would not
      // move the reference and the row max is not needed (the result is the same
      // bit for bit).  Otherwise, or before the first reference, the warp
      // reloads S and takes the rule.
      float alpha = 1.f, sum = 0.f;
      bool full = m_ref == -CUDART_INF_F;
      const bool tried = !__any_sync(0xffffffffu, full);
      if (tried) {
        sum = row_exp_n<KT>(s, sl2, m_ref * sl2);
        full = !(sum <= 256.f);
      }
      if (__any_sync(0xffffffffu, full)) {
        if (tried) load_s();  // the attempt overwrote s
        const float mx = row_max_n<KT>(s);
        if (mx != -CUDART_INF_F &&
            (m_ref == -CUDART_INF_F || (mx - m_ref) * sl2 > kRescaleLog2)) {
          alpha = m_ref == -CUDART_INF_F ? 0.f : ex2_approx((m_ref - mx) * sl2);
          m_ref = mx;
        }
        const float mu = m_ref == -CUDART_INF_F ? 0.f : m_ref * sl2;
        sum = row_exp_n<KT>(s, sl2, mu);  // masked: 2^-inf = 0
      }
      l = fmaf(l, alpha, sum);
      {
        uint32_t w[KT / 2];
#pragma unroll
        for (int c = 0; c < KT / 2; ++c) w[c] = Pack2<T>::run(s[2 * c], s[2 * c + 1]);
        if constexpr (KT == 32) {
          tmem_st16u(t_s, w);  // P over the first 16 columns of S
        } else {
          tmem_st32u(t_s, w);
        }
      }
      // rescale this warp's O rows once P.V(j - 1) has finished with them
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        if (!wait_phase(smem_u32(&bar_o[(j - 1) & 1]), ((j - 1) >> 1) & 1)) fail = true;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (!__any_sync(0xffffffffu, fail)) {
          // 16 columns at a time (32 would spill under this kernel's register bound)
#pragma unroll
          for (int cb = 0; cb < D; cb += 16) {
            uint32_t o[16];
            tmem_ld16u(t_o + cb, o);
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st16u(t_o + cb, o);
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();  // the warp's P (and O) stores are done
      if (lane == 0) mbar_arrive(&bar_p[j & 1]);
      if (__any_sync(0xffffffffu, fail)) {
        fail = true;
        break;
      }
    }
    // the last P.V
    if (ntiles > 0 && !fail &&
        !wait_phase(smem_u32(&bar_o[(ntiles - 1) & 1]), ((ntiles - 1) >> 1) & 1))
      fail = true;
  }

  // ---- results (after every role has stopped) ------------------------------
  if (fail) s_fail = 1;
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // every role is done; s_bad and s_fail are final
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  pdl_trigger();
  if (warp_live) {
    const uint32_t t_o = tmem + 2 * KT + (static_cast<uint32_t>(warp * 32) << 16);
    const bool failed = s_fail != 0;
    const bool bad = bad_len || s_bad != 0 || failed;
    const bool have_o = ntiles > 0 && !failed;  // uniform over the CTA
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
        tmem_ld32(t_o + cb, o);  // warp-collective: every lane of a live warp loads
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
  }
  if (tid == 0 && s_fail != 0) report_error(p.dev_err, PA_DEV_TIMEOUT);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // every tensor-memory load of the results is done
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(S::kTmemCols));
  }
}

template <typename T, int D>
cudaError_t launch_d(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  auto kern = chunk_tc_pipe_kernel<T, D>;
  constexpr int KT = PipeShape<D>::kKeyTile;
  const int smem = PipeSizes<D>::kSmem;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  // tensor-map copies need pages of at least 8 tokens (a 1024-byte swizzle
  // atom per copy); otherwise, or without an encoder, every tile uses cp.async
  CUtensorMap mk{}, mv{};
  const int use_tma = p.block_size_log2 >= 3 && pool_tensor_map(&mk, p.k_pool, dtype, p, KT) &&
                      pool_tensor_map(&mv, p.v_pool, dtype, p, KT);
  const int nblk = (p.chunk_len * p.group + kRows - 1) / kRows;
  dim3 grid(nblk * p.num_kv_heads, p.num_seqs, p.partial_out ? p.num_splits : 1);
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, p, mk, mv, use_tma,
                    withhold_tiles());
}

template <typename T>
cudaError_t launch_t(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (p.head_dim == 64) return launch_d<T, 64>(p, dtype, stream);
  if (p.head_dim == 128) return launch_d<T, 128>(p, dtype, stream);
  return cudaErrorInvalidValue;
}

}  // namespace

// Every chunk past the decode kernel's chunk mode (16 columns at head_dim 64, 8
// at 128) and below two Q tiles.  It replaced the mma.sync chunk kernel below 64
// (head_dim 64) and 128 (head_dim 128) rows, and a one-tile tcgen05 kernel that
// ran each key tile's phases in order above: at head_dim 64, 24 / 32 / 48 / 64
// rows (6 / 8 / 12 / 16 queries of the 64 x 4096-token batch) took 104.4 / 104.7
// / 106.8 / 107.8 us against 115.3 / 116.4 / 137.2 / 129.2; at head_dim 128, the
// 8 x 32,768-token batch in 64-page splits took 227 / 256 / 281 / 308 us at 4 / 16
// / 24 / 32 queries against 238 / 297 / 550 / 344, one pass of 32 queries 810
// against 992 us.
bool chunk_tc_pipe_supports(pa_dtype dtype, int head_dim, int rows) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  if (head_dim == 128) return rows >= 9;
  return head_dim == 64 && rows >= 17;
}

cudaError_t launch_chunk_tc_pipe(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_t<__nv_bfloat16>(p, dtype, stream);
  if (dtype == PA_F16) return launch_t<__half>(p, dtype, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
