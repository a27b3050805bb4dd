// Warp-specialized chunked read / prefill on the tcgen05 tensor cores.
//
// Same contract as the other chunk reads (nanoserve "Day 23: the real
// triton.jit paged-attention kernel": query i of a chunk sits at position
// past + i and sees tokens 0 .. past + i), same per-row arithmetic as
// chunk_tc_kernel (fp32 online softmax with a lazily moved reference max,
// P rounded to the cache dtype), but the phases of a key tile run on
// different warps at the same time instead of one after the other:
//
//   warps 0, 3   load, alternately, 64-token K/V tiles through the block
//                table ("Three Attention Kernels", section "3. Paged KV-cache
//                attention") into a 4-stage ring: a tile whose tokens all
//                exist by 2D tensor-map copies (cp.async.bulk.tensor, one per
//                page and head_dim half, counted in bytes on the stage's
//                `full` mbarrier); the last tile of a range (or pages of
//                fewer than 8 tokens) by 16-byte cp.async with zero-fill,
//                announced once the warp's own copies have landed
//   warps 1, 2   MMA: lane 0 of warp 1 + k issues S_k = Q_k . K^T and
//                O_k += P_k . V for Q tile k (tcgen05.mma, fp32 accumulators
//                in tensor memory) and commits each to an mbarrier; QK(j + NB)
//                goes right after P.V(j), into the S buffer P.V(j) has read
//                (NB = 3 S buffers per Q tile at head_dim 64, 2 at 128)
//   warps 4-7    softmax of Q tile 0, warps 8-11 of Q tile 1: thread r of a
//                group owns row r (tensor-memory lane r), reads its S row,
//                writes its P row back over S as 16-bit pairs, and moves
//                the reference max (rescaling its O row) only when a score
//                passes it by more than 2^8
//
// While the softmax warps of one Q tile work on key tile j, S(j + 1) (and at
// head_dim 64 S(j + 2)) is already in tensor memory, the tensor core runs the other products, and
// the load warps fetch the next tiles.  Two Q tiles share every K/V tile, so
// each copy feeds twice the math.
//
// Tensor memory: S_0[0..NB-1] | S_1[0..NB-1] (64 columns each) | O_0 | O_1
// (head_dim each): 512 columns at head_dim 64 (NB 3) and at 128 (NB 2).
// mbarriers: full/empty per ring stage, and per Q tile and
// S buffer s (S ready), p (P written, one arrival per softmax warp), o (P.V
// done: the buffer and O free again); at head_dim 128 also one per softmax
// group for taking turns at the exponentials.  One barrier per buffer means
// no waiter can see a barrier complete twice before it looks (parity waits
// would misread that).  Every wait is bounded (about a second); on time-out
// the kernel records PA_DEV_TIMEOUT, every role leaves its loop, the outputs
// are zeroed and the tensor memory is freed.
#include <cuda.h>  // CUtensorMap (the encoder is fetched through the runtime)
#include <math_constants.h>

#include <atomic>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tc.cuh"

namespace pa {
namespace {

using namespace tc;

constexpr int kQRows = 128;                  // rows of one Q tile (the MMA M)
constexpr int kQTiles = 2;                   // Q tiles per CTA
constexpr int kCtaRows = kQRows * kQTiles;
constexpr int kKeyTile = 64;                 // tokens per K/V tile
constexpr int kThreads = 384;                // 12 warps
constexpr int kAllocWarp = 2, kSoftmaxWarp0 = 4;
constexpr int kLoaders = 2;                  // warps 0 and 3 load tiles j = 0, 1 (mod 2)
// warps 1 and 2 issue the MMAs of Q tiles 0 and 1: one thread's tcgen05.mma
// issue takes ~100+ cycles, so two issuers keep the tensor pipe about twice as busy
constexpr float kRescaleLog2 = 8.f;

// S buffers per Q tile and K/V ring stages at head_dim 64 (see WsShape)
#ifndef PA_WS_SBUF_D64
#define PA_WS_SBUF_D64 3
#endif
#ifndef PA_WS_STAGES_D64
#define PA_WS_STAGES_D64 6
#endif

template <int D>
struct WsShape {
  static constexpr int kQBytes = kQRows * D * 2;     // one Q tile: [kb][128 rows][128 B]
  static constexpr int kKVBytes = kKeyTile * D * 2;  // one K or V tile: [kb][64 rows][128 B]
  // K/V ring depth: QK(j + kSBuf) needs key tile j + kSBuf, whose stage was released by
  // P.V(j + kSBuf - kStages); the stages beyond kSBuf are the loads' time to arrive.
  // 6 stages at head_dim 64 (16 KB each, 129 KB with Q), 4 at 128 (32 KB each, 193 KB).
  // Same-GPU A/B at head_dim 64 (S buffers x stages, prefill 8 x 4096 / 64-query chunks
  // at history 4096, us): 2 x 4 848 / 231, 2 x 8 856 / 224, 3 x 8 852 / 223,
  // 3 x 6 846 / 223; 3 buffers with 4 stages took 922 / 301 (the key loads then sit on
  // the critical path).
  static constexpr int kStages = D <= 64 ? PA_WS_STAGES_D64 : 4;
  static constexpr int kSmem = kQTiles * kQBytes + kStages * 2 * kKVBytes + 1024;
  // S_k in kSBuf buffers per Q tile (tile j in buffer j % kSBuf), then O_k.  Three
  // buffers at head_dim 64 (3 * 2 * 64 + 2 * 64 = 512 columns, all of tensor memory),
  // two at 128: QK(j + kSBuf) can only overwrite the buffer P.V(j) has finished
  // reading, so the chain softmax(j) -> P.V(j) -> QK(j + kSBuf) -> softmax(j + kSBuf)
  // spreads over kSBuf tiles.
  static constexpr int kSBuf = D <= 64 ? PA_WS_SBUF_D64 : 2;
  static constexpr int kSCols = kQTiles * kSBuf * kKeyTile;
  static constexpr int kTmemUsed = kSCols + kQTiles * D;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    chunk_tc_ws_kernel(const ChunkParams p, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v, const int use_tma,
                       const int withhold) {
  using S = WsShape<D>;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  constexpr int NB = S::kSBuf;
  constexpr int kStages = S::kStages;
  __shared__ uint64_t bar_full[kStages], bar_empty[kStages];
  __shared__ uint64_t bar_s[kQTiles][NB], bar_p[kQTiles][NB], bar_o[kQTiles][NB];
  __shared__ uint64_t bar_turn[kQTiles];  // softmax groups take turns at the exponentials
  __shared__ uint32_t tmem_base;
  __shared__ int s_bad, s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hkv = p.num_kv_heads, G = p.group, nq = p.chunk_len;
  const int g = blockIdx.x % hkv;
  const int rows_total = nq * G;
  const int nblk = (rows_total + kCtaRows - 1) / kCtaRows;
  const int rblk = nblk - 1 - blockIdx.x / hkv;  // the longest causal ranges start first
  const int b = blockIdx.y;
  const int split = blockIdx.z;
  const bool partial = p.partial_out != nullptr;
  const int bs_log2 = p.block_size_log2, bs_mask = (1 << bs_log2) - 1;

  unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  unsigned char *sq = smem;                          // Q tile 0, Q tile 1
  unsigned char *skv = smem + kQTiles * S::kQBytes;  // stage st: K at 2*st, V at 2*st + 1

  if (tid == 0) {
    s_bad = 0;
    s_fail = 0;
#pragma unroll
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], kQTiles);  // released by both MMA warps
    }
#pragma unroll
    for (int k = 0; k < kQTiles; ++k) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        mbar_init(&bar_s[k][nb], 1);
        mbar_init(&bar_p[k][nb], kQRows / 32);  // one arrival per softmax warp
        mbar_init(&bar_o[k][nb], 1);
      }
      mbar_init(&bar_turn[k], kQRows / 32);
    }
  }
  if (warp == kAllocWarp) {
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
  // key tiles of each Q tile (its last row's causal limit), and of the CTA
  const int base0 = rblk * kCtaRows;
  int nt[kQTiles];
  int kv_end = t_lo;
#pragma unroll
  for (int k = 0; k < kQTiles; ++k) {
    const int base = base0 + k * kQRows;
    if (base >= rows_total) {
      nt[k] = 0;
    } else {
      const int last = min(rows_total - 1, base + kQRows - 1);
      const int end = max(t_lo, min(t_hi, past + last / G + 1));
      nt[k] = (end - t_lo + kKeyTile - 1) / kKeyTile;
      kv_end = max(kv_end, end);
    }
  }
  const int ntiles = max(nt[0], nt[1]);

  // ---- both Q tiles into the swizzled K-major layout (all threads) --------
  const T *qbase = static_cast<const T *>(p.q);
  for (int idx = tid; idx < kCtaRows * (D / 8); idx += kThreads) {
    const int r = idx / (D / 8), c = idx - r * (D / 8);
    const int qr = base0 + r;
    const bool ok = qr < rows_total;
    const T *src = qbase;
    if (ok) {
      const int i = qr / G, h = qr - (qr / G) * G;
      src = qbase + ((static_cast<size_t>(b) * nq + i) * p.num_q_heads +
                     static_cast<size_t>(g) * G + h) * D + c * 8;
    }
    cp_async16(sq + (r / kQRows) * S::kQBytes + sw_off(r % kQRows, c, kQRows), src, ok);
  }
  cp_async_commit();
  cp_async_wait_all();
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // barriers, tensor-memory address, Q
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  bool fail = false;

  // softmax-warp state: Q tile k_sm, tensor-memory lanes 32*quad .. 32*quad+31,
  // one row per thread (unused by the other warps)
  const bool is_softmax = warp >= kSoftmaxWarp0;
  const int k_sm = is_softmax ? (warp - kSoftmaxWarp0) >> 2 : 0;
  const int quad = warp & 3;
  const int row = base0 + k_sm * kQRows + quad * 32 + lane;
  const bool row_ok = is_softmax && row < rows_total;
  const bool warp_live = is_softmax && base0 + k_sm * kQRows + quad * 32 < rows_total;
  const int my_nt = is_softmax ? (k_sm == 0 ? nt[0] : nt[1]) : 0;
  const uint32_t t_lane = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t t_s0 = tmem + k_sm * NB * kKeyTile + t_lane;  // S buffer 0; buffer b at +64 b
  const uint32_t t_o = tmem + S::kSCols + k_sm * D + t_lane;
  const float sl2 = fmaxf(fabsf(p.scale_log2), 1e-30f);
  float m_ref = -CUDART_INF_F;  // reference max (raw units) of the exponent
  float l = 0.f;

  const int loader = warp == 0 ? 0 : warp == 3 ? 1 : -1;
  const int mma_k = warp == 1 ? 0 : warp == 2 ? 1 : -1;
  if (loader >= 0) {
    // ---------------------------------------------------------- load warps
    // Loader w fetches tiles j = w, w + 2, ...: waits for its ring stage to be
    // released and copies the tile (page ids read and checked one of its tiles
    // ahead).  A tile whose 64 tokens all exist goes through the tensor maps:
    // lane 0 issues one 2D copy per page and head_dim half, counted in bytes
    // on the stage's `full` barrier, and moves on.  A tile that runs past the
    // end (or pages of fewer than 8 tokens) is copied by the warp with 16-byte
    // cp.async and zero-fill, so that no stale row can reach P.V; the warp
    // waits for those copies and then announces the tile.
    const int32_t *bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks;
    const T *kpool = static_cast<const T *>(p.k_pool);
    const T *vpool = static_cast<const T *>(p.v_pool);
    // page ids of tile j's pages (at most 64: one token per page), lane l
    // holding pages first + l and first + 32 + l; an id outside the pool is
    // reported, marks the CTA's outputs bad and reads as -1 (no copy)
    auto fetch_pages = [&](int j, int &pa, int &pb) {
      pa = pb = -1;
      if (j < ntiles) {
        const int t0 = t_lo + j * kKeyTile;
        const int first = t0 >> bs_log2;
        const int last = (min(t0 + kKeyTile, kv_end) - 1) >> bs_log2;  // < max_blocks
        if (first + lane <= last) pa = __ldg(bt_row + first + lane);
        if (first + 32 + lane <= last) pb = __ldg(bt_row + first + 32 + lane);
        const bool bad_a = first + lane <= last && (pa < 0 || pa >= p.num_pages);
        const bool bad_b = first + 32 + lane <= last && (pb < 0 || pb >= p.num_pages);
        if (bad_a || bad_b) {
          report_error(p.dev_err, PA_DEV_BAD_PAGE);
          s_bad = 1;
          if (bad_a) pa = -1;
          if (bad_b) pb = -1;
        }
      }
    };
    int pa, pb;
    fetch_pages(loader, pa, pb);
    // test hook: no tile is ever announced, so the other roles' waits run out
    for (int j = loader; j < ntiles && !withhold; j += kLoaders) {
      const int st = j % kStages;
      if (j >= kStages && !wait_phase(smem_u32(&bar_empty[st]), ((j / kStages) - 1) & 1)) {
        fail = true;
        break;
      }
      unsigned char *ks = skv + (2 * st) * S::kKVBytes;
      unsigned char *vs = ks + S::kKVBytes;
      const int t0 = t_lo + j * kKeyTile;
      const int first = t0 >> bs_log2;
      int na, nb;
      fetch_pages(j + kLoaders, na, nb);
      if (use_tma && t0 + kKeyTile <= kv_end) {
        // pages of the tile: 64 / bs of them (bs < 64), or one 64-row part of a page
        const int rows = bs_log2 >= 6 ? kKeyTile : (1 << bs_log2);
        const int npg = kKeyTile / rows;  // <= 8 (bs >= 8)
        int pg[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pg[i] = __shfl_sync(0xffffffffu, pa, i);  // lane i < npg
        if (lane == 0) {
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (i < npg && pg[i] >= 0) bytes += 2u * rows * D * 2u;
          mbar_arrive_expect(&bar_full[st], bytes);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if (i >= npg || pg[i] < 0) continue;  // a bad page: the outputs are zeroed anyway
            const int y = (pg[i] << bs_log2) + (bs_log2 >= 6 ? (t0 & bs_mask) : 0);
#pragma unroll
            for (int kb = 0; kb < D / 64; ++kb) {
              const uint32_t off = kb * (kKeyTile * 128) + i * rows * 128;
              tma_load_2d(ks + off, &tmap_k, g * D + kb * 64, y, &bar_full[st]);
              tma_load_2d(vs + off, &tmap_v, g * D + kb * 64, y, &bar_full[st]);
            }
          }
        }
        __syncwarp();
        pa = na;
        pb = nb;
        continue;
      }
#pragma unroll 4
      for (int idx = lane; idx < kKeyTile * (D / 8); idx += 32) {
        const int tr = idx / (D / 8), c = idx % (D / 8);
        const int t = t0 + tr;
        const int pi = (t >> bs_log2) - first;  // 0 .. 63
        const int pg_a = __shfl_sync(0xffffffffu, pa, pi & 31);
        const int pg_b = __shfl_sync(0xffffffffu, pb, pi & 31);
        const int page = pi < 32 ? pg_a : pg_b;
        const bool valid = t < kv_end && page >= 0;
        const size_t off =
            valid ? (((static_cast<size_t>(page) << bs_log2) + (t & bs_mask)) * hkv + g) * D + c * 8
                  : 0;
        const uint32_t o = sw_off(tr, c, kKeyTile);
        cp_async16(ks + o, kpool + off, valid);
        cp_async16(vs + o, vpool + off, valid);
      }
      cp_async_commit();
      pa = na;
      pb = nb;
      cp_async_wait_all();
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_full[st]);
    }
    cp_async_wait_all();
  } else if (mma_k >= 0) {
    // ---------------------------------------------------------- MMA warps
    // Warp 1 + k issues Q tile k's products: QK(0) .. QK(NB - 1), then for each
    // tile j: P.V(j), release of stage j, and QK(j + NB) into the S buffer
    // P.V(j) has just read.  So S(j + 1) is ready while the softmax works on
    // tile j, and the softmax warps do not wait for the tensor core.
    if (lane == 0) {
      const int k = mma_k;
      const uint32_t id_qk = idesc<T>(kQRows, kKeyTile, false, p.scale_log2 < 0.f);
      const uint32_t id_pv = idesc<T>(kQRows, D, true, false);
      const uint32_t qs_u = smem_u32(sq + k * S::kQBytes);
      const uint32_t t_o_k = tmem + S::kSCols + k * D;
      // S_k[j % NB] = Q_k . K_j^T, once tile j is in and the buffer is free (P_k
      // of tile j - NB has gone through P.V: completion (j - NB) / NB of its
      // barrier, the last one it can have had, since P.V(j) needs this S)
      auto issue_qk = [&](int j) -> bool {
        if (!wait_phase(smem_u32(&bar_full[j % kStages]), (j / kStages) & 1)) return false;
        if (j >= NB && !wait_phase(smem_u32(&bar_o[k][j % NB]), ((j / NB) - 1) & 1)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t ks_u = smem_u32(skv + (2 * (j % kStages)) * S::kKVBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
          mma_f16(tmem + (NB * k + (j % NB)) * kKeyTile,
                  sw128_desc(qs_u + kb * (kQRows * 128) + kin, 16, 1024),
                  sw128_desc(ks_u + kb * (kKeyTile * 128) + kin, 16, 1024), id_qk, ks > 0);
        }
        commit(smem_u32(&bar_s[k][j % NB]));
        return true;
      };
      // O_k += P_k . V_j once the softmax warps of Q tile k have written P_k
      auto issue_pv = [&](int j) -> bool {
        if (!wait_phase(smem_u32(&bar_p[k][j % NB]), (j / NB) & 1)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t vs_u = smem_u32(skv + (2 * (j % kStages) + 1) * S::kKVBytes);
        const uint32_t t_s = tmem + (NB * k + (j % NB)) * kKeyTile;
#pragma unroll
        for (int kk = 0; kk < kKeyTile / 16; ++kk)
          mma_f16_ta(t_o_k, t_s + kk * 8, sw128_desc(vs_u + kk * 2048, kKeyTile * 128, 1024),
                     id_pv, (j > 0 || kk > 0));
        commit(smem_u32(&bar_o[k][j % NB]));
        return true;
      };
      const int my = k == 0 ? nt[0] : nt[1];
      for (int j = 0; j < NB && j < my && !fail; ++j)
        if (!issue_qk(j)) fail = true;
      for (int j = 0; j < my && !fail; ++j) {
        if (!issue_pv(j)) {
          fail = true;
          break;
        }
        commit(smem_u32(&bar_empty[j % kStages]));  // stage j is free once P.V(j) is done
        if (j + NB < my && !issue_qk(j + NB)) fail = true;
      }
      // tiles this Q tile does not need: release each after it arrived, so that
      // a stage is never released ahead of its fill
      for (int j = my; j < ntiles && !fail; ++j) {
        if (!wait_phase(smem_u32(&bar_full[j % kStages]), (j / kStages) & 1)) {
          fail = true;
          break;
        }
        commit(smem_u32(&bar_empty[j % kStages]));
      }
      // the loaders do not wait for the last stages' releases: wait for them
      // here, so no arrival reaches this CTA's shared memory after it exits
      for (int j = max(0, ntiles - kStages); j < ntiles && !fail; ++j)
        if (!wait_phase(smem_u32(&bar_empty[j % kStages]), (j / kStages) & 1)) fail = true;
    }
    __syncwarp();
  } else if (is_softmax) {
    // ---------------------------------------------------------- softmax warps
    const int k = k_sm;
    const int pos = min(past + row / G, t_hi - 1);  // this row's last key (inclusive)
    // At head_dim 128 the two groups take turns at the row max and
    // exponentials of the tiles both Q tiles read (group 0 first), so each
    // runs them with the exp unit of its SMSP to itself while the other loads
    // S or stores P (at head_dim 64, with half the MMA time per tile to
    // overlap, taking turns measured slower).  Group k
    // waits on bar_turn[k]: group 0 for group 1's tile j - 1, group 1 for
    // group 0's tile j.  Either barrier's next completion needs its waiter's
    // own progress, so a parity wait never sees two completions.
    const int n_pair = (nt[0] > 0 && nt[1] > 0) ? min(nt[0], nt[1]) : 0;
    for (int j = 0; j < my_nt; ++j) {
      if (!wait_phase(smem_u32(&bar_s[k][j % NB]), (j / NB) & 1)) {
        fail = true;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t t_s = t_s0 + (j % NB) * kKeyTile;
      const int tok0 = t_lo + j * kKeyTile;
      float s[kKeyTile];
      // S row of this thread, -inf past its last key
      auto load_s = [&]() {
        tmem_ld64(t_s, s);
        if (tok0 + kKeyTile - 1 > pos) {  // the tile crosses this row's last key
#pragma unroll
          for (int c = 0; c < kKeyTile; ++c)
            if (tok0 + c > pos) s[c] = -CUDART_INF_F;
        }
      };
      if (warp_live) load_s();
      const bool turns = D > 64 && j < n_pair;
      if (turns && (k == 1 || j > 0) &&
          !wait_phase(smem_u32(&bar_turn[k]), (k == 0 ? j - 1 : j) & 1))
        fail = true;
      float alpha = 1.f;
      if (warp_live && !fail) {
        float sum = 0.f;
        bool full = true;  // take the lazy rule (and the row max)
        if constexpr (D == 64) {
          // Common case first: exponents against the current reference.  When
          // their sum is at most 2^8 no probability exceeds 2^8, so the rule
          // would not move the reference and the row max is not needed.
          // Otherwise (or on a first tile) the warp reloads S and takes the
          // rule.  (At head_dim 128, with its registers nearly all in use, the
          // extra path measured slower.)
          full = j == 0 || m_ref == -CUDART_INF_F;
          if (!__any_sync(0xffffffffu, full)) {
            sum = row_exp64(s, sl2, m_ref * sl2);
            full = !(sum <= 256.f);
          }
          full = __any_sync(0xffffffffu, full);
          if (full && j > 0) load_s();  // the fast attempt overwrote s (warp-collective)
        }
        if (full) {
          // the lazy rule: the reference max moves only when a score passes it
          // by more than 2^8
          const float mx = row_max64(s);
          if (mx != -CUDART_INF_F &&
              (m_ref == -CUDART_INF_F || (mx - m_ref) * sl2 > kRescaleLog2)) {
            alpha = m_ref == -CUDART_INF_F ? 0.f : ex2_approx((m_ref - mx) * sl2);
            m_ref = mx;
          }
          const float mu = m_ref == -CUDART_INF_F ? 0.f : m_ref * sl2;
          sum = row_exp64(s, sl2, mu);  // masked: 2^-inf = 0
        }
        l = fmaf(l, alpha, sum);
      }
      if (turns) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_turn[1 - k]);
      }
      if (warp_live && !__any_sync(0xffffffffu, fail)) {
        {
          uint32_t w[kKeyTile / 2];
#pragma unroll
          for (int c = 0; c < kKeyTile / 2; ++c) w[c] = Pack2<T>::run(s[2 * c], s[2 * c + 1]);
          tmem_st32u(t_s, w);  // P over the first 32 columns of S
        }
        // rescale this warp's O rows once the previous P.V has finished with them
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!wait_phase(smem_u32(&bar_o[k][(j - 1) % NB]), ((j - 1) / NB) & 1)) fail = true;
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          if (!__any_sync(0xffffffffu, fail)) {
#pragma unroll
            for (int cb = 0; cb < D; cb += 32) {
              float o[32];
              tmem_ld32(t_o + cb, o);
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] *= alpha;
              tmem_st32(t_o + cb, o);
            }
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();  // the warp's P (and O) stores are done
      if (lane == 0) mbar_arrive(&bar_p[k][j % NB]);
      if (__any_sync(0xffffffffu, fail)) {
        fail = true;
        break;
      }
    }
    // the last P.V of this Q tile
    if (my_nt > 0 && !fail &&
        !wait_phase(smem_u32(&bar_o[k][(my_nt - 1) % NB]), ((my_nt - 1) / NB) & 1))
      fail = true;
  }

  // ---- results (after every role has stopped) ------------------------------
  if (fail) s_fail = 1;
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();  // every role is done; s_bad and s_fail are final
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  pdl_trigger();
  if (is_softmax) {
    const bool failed = s_fail != 0;
    const bool bad = bad_len || s_bad != 0 || failed;
    const bool have_o = my_nt > 0 && !failed;  // uniform over the warp
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
    if (partial && row_ok)
      p.partial_lse[prow] =
          empty ? -CUDART_INF_F : fmaf(m_ref, sl2, log2f(l)) * 0.69314718055994531f;
#pragma unroll
    for (int cb = 0; cb < D; cb += 32) {
      float o[32];
      if (have_o && warp_live) {
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
  if (warp == kAllocWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(S::kTmemCols));
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the CUDA driver's tensor-map encoder, looked up once (null if unavailable)
EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(f);
  });
  return fn;
}

// A 2D view of a pool: rows = num_pages * block_size token rows of Hkv * D
// elements; a box is 64 elements (one 128-byte swizzle span) by
// min(block_size, box_rows) rows, so one copy moves one kv head's rows of a
// page (or of a key tile's part of a page).
bool make_pool_map(CUtensorMap *map, const void *pool, pa_dtype dtype, const ChunkParams &p,
                   int box_rows) {
  EncodeTiled enc = encoder();
  if (enc == nullptr) return false;
  const int bs = 1 << p.block_size_log2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.num_kv_heads) * p.head_dim,
                              static_cast<cuuint64_t>(p.num_pages) * bs};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.num_kv_heads) * p.head_dim * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(bs < box_rows ? bs : box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map,
                         dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                          : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                         2, const_cast<void *>(pool), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Recently encoded pool maps, so that a serving loop calling with the same
// pools encodes each map once.  A map is a pure function of its arguments
// (the pool's address, extents and dtype), valid in any context.
struct MapKey {
  const void *pool;
  int32_t num_pages, block_size_log2, num_kv_heads, head_dim, box_rows;
  pa_dtype dtype;
  bool operator==(const MapKey &o) const {
    return pool == o.pool && num_pages == o.num_pages && block_size_log2 == o.block_size_log2 &&
           num_kv_heads == o.num_kv_heads && head_dim == o.head_dim && box_rows == o.box_rows &&
           dtype == o.dtype;
  }
};
constexpr int kMapCache = 16;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_used = 0, g_map_next = 0;

}  // namespace

bool pool_tensor_map(CUtensorMap *map, const void *pool, pa_dtype dtype, const ChunkParams &p,
                     int box_rows) {
  const MapKey key{pool, p.num_pages, p.block_size_log2, p.num_kv_heads, p.head_dim, box_rows,
                   dtype};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_key[i] == key) {
        *map = g_map_val[i];
        return true;
      }
  }
  if (!make_pool_map(map, pool, dtype, p, box_rows)) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  const int i = g_map_used < kMapCache ? g_map_used++ : (g_map_next++ % kMapCache);
  g_map_key[i] = key;
  g_map_val[i] = *map;
  return true;
}

// Test hook for the time-out path (set through pa_test_set_withhold_tiles):
// the load warps announce no tile, every wait then runs out (after about a
// second of the global timer, or 2^26 polls) and the call reports
// PA_DEV_TIMEOUT with zeroed outputs.  Nothing is in flight when the waits
// give up.  Off unless a test turns it on.
std::atomic<int> g_withhold_tiles{0};

int withhold_tiles() { return g_withhold_tiles.load(std::memory_order_relaxed); }

namespace {

template <typename T, int D>
cudaError_t launch_d(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  auto kern = chunk_tc_ws_kernel<T, D>;
  const int smem = WsShape<D>::kSmem;
  cudaError_t err = set_max_smem(reinterpret_cast<const void *>(kern), smem);
  if (err != cudaSuccess) return err;
  // tensor-map copies need pages of at least 8 tokens (a 1024-byte swizzle
  // atom per copy); otherwise, or without an encoder, every tile uses cp.async
  CUtensorMap mk{}, mv{};
  const int use_tma = p.block_size_log2 >= 3 &&
                      pool_tensor_map(&mk, p.k_pool, dtype, p, kKeyTile) &&
                      pool_tensor_map(&mv, p.v_pool, dtype, p, kKeyTile);
  const int withhold = withhold_tiles();
  const int nblk = (p.chunk_len * p.group + kCtaRows - 1) / kCtaRows;
  dim3 grid(nblk * p.num_kv_heads, p.num_seqs, p.partial_out ? p.num_splits : 1);
  return launch_pdl(kern, grid, dim3(kThreads), smem, stream, p, mk, mv, use_tma, withhold);
}

template <typename T>
cudaError_t launch_t(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  switch (p.head_dim) {
    case 64: return launch_d<T, 64>(p, dtype, stream);
    case 128: return launch_d<T, 128>(p, dtype, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

bool chunk_tc_ws_supports(pa_dtype dtype, int head_dim, int rows) {
  if (dtype != PA_F16 && dtype != PA_BF16) return false;
  if (head_dim != 64 && head_dim != 128) return false;
  return rows >= kCtaRows;
}

cudaError_t launch_chunk_tc_ws(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (dtype == PA_BF16) return launch_t<__nv_bfloat16>(p, dtype, stream);
  if (dtype == PA_F16) return launch_t<__half>(p, dtype, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa

extern "C" void pa_test_set_withhold_tiles(int32_t on) {
  pa::g_withhold_tiles.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
}
