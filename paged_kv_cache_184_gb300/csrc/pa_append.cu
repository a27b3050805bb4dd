// Cache append: scatter each new token's K and V row into its page slot.
//
// nanoserve "Day 20: the number the Triton kernel has to beat", section
// "What I learned": the write grows the block table and scatters the K/V.
// The caller grows the table; this kernel is the scatter.  A token row is
// the contiguous [num_kv_heads][head_dim] slice at one slot of one page, so
// every thread moves one aligned 16-byte chunk of K and one of V: a plain
// byte copy, bit-exact.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) append_kernel(const AppendParams p) {
  pdl_trigger();  // the read that follows may launch now; it waits for this grid
  pdl_wait();
  const long long gid = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  const long long total = static_cast<long long>(p.num_tokens) * p.row_chunks;
  if (gid >= total) return;
  const int i = static_cast<int>(gid / p.row_chunks);
  const int c = static_cast<int>(gid - static_cast<long long>(i) * p.row_chunks);

  const int seq = p.seq_ids != nullptr ? p.seq_ids[i] : i;
  if (seq < 0 || seq >= p.num_seqs) {
    report_error(p.dev_err, PA_DEV_BAD_SEQ_ID);
    return;
  }
  const int pos = p.positions[i];
  const long long cap = static_cast<long long>(p.max_blocks) << p.block_size_log2;
  if (pos < 0 || static_cast<long long>(pos) >= cap) {
    report_error(p.dev_err, PA_DEV_BAD_POSITION);
    return;
  }
  const int page = p.block_table[static_cast<size_t>(seq) * p.max_blocks + (pos >> p.block_size_log2)];
  if (page < 0 || page >= p.num_pages) {
    report_error(p.dev_err, PA_DEV_BAD_PAGE);
    return;
  }
  const size_t row = (static_cast<size_t>(page) << p.block_size_log2) +
                     (pos & ((1 << p.block_size_log2) - 1));
  const size_t src = static_cast<size_t>(i) * p.row_chunks + c;
  const size_t dst = row * p.row_chunks + c;
  const uint4 kv = __ldg(static_cast<const uint4 *>(p.k_new) + src);
  const uint4 vv = __ldg(static_cast<const uint4 *>(p.v_new) + src);
  static_cast<uint4 *>(p.k_pool)[dst] = kv;
  static_cast<uint4 *>(p.v_pool)[dst] = vv;
}

}  // namespace

cudaError_t launch_append(const AppendParams &p, cudaStream_t stream) {
  const long long total = static_cast<long long>(p.num_tokens) * p.row_chunks;
  const long long blocks = (total + kThreads - 1) / kThreads;
  return launch_pdl(append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), 0, stream,
                    p);
}

}  // namespace pa
