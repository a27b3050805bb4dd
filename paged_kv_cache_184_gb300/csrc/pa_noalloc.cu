// pa_decode_splitkv_noalloc: the split-KV read and its merge in one call,
// for callers that cannot allocate device memory.
//
// The split read needs somewhere to put its per-split partial outputs and
// log-sum-exps before the merge combines them.  pa_decode_splitkv takes that
// space from the caller.  Some callers have no way to provide it: a plugin
// running inside a host framework that owns every device allocation (and
// hands the plugin only its inputs and outputs), or a latency-critical
// serving loop that must never call cudaMalloc/cudaFree because they can
// synchronize the whole device.  This entry point keeps the partials in a
// fixed array that the library itself places in device memory when it is
// loaded, so a call allocates nothing.
//
// The array is shared by every call on a device and keeps whatever the last
// call left in it.  Nothing here depends on its earlier contents: the split
// read writes every partial (including -inf for empty splits) that the merge
// then reads.  Two calls whose kernels overlap on the GPU (on different
// streams, or from different host threads) use the same array and race.
#include <mutex>

#include "pa_internal.h"

namespace {

// Lives in device memory on every GPU that loads the library, until exit.
__device__ __align__(256) unsigned char g_partials[PA_NOALLOC_SCRATCH_BYTES];

// Device addresses of g_partials found so far, one per CUDA context.  The
// address belongs to the context the module was loaded into, not to the
// device ordinal: after a device reset (or in another context on the same
// device) the module is loaded again and the array may sit elsewhere.  The
// key is the driver's context id, unique for the life of the process, so an
// address found in one context is never used in another.
struct Known {
  uint64_t ctx;
  unsigned char *addr;
};
constexpr int kKnown = 64;
std::mutex g_known_mu;
Known g_known[kKnown];
int g_known_used = 0, g_known_next = 0;

// Device address of g_partials in the current context (in host code the
// symbol itself is only a host-side handle).  The first call in a context
// looks it up with cudaGetSymbolAddress; later calls in that context reuse
// it.  Without a readable context id every call looks it up.
cudaError_t partials_address(unsigned char **addr) {
  const uint64_t ctx = pa::current_context_id();
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_known_mu);
    for (int i = 0; i < g_known_used; ++i)
      if (g_known[i].ctx == ctx) {
        *addr = g_known[i].addr;
        return cudaSuccess;
      }
  }
  void *sym = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&sym, g_partials);
  if (err != cudaSuccess) return err;
  *addr = static_cast<unsigned char *>(sym);
  if (ctx != 0) {
    std::lock_guard<std::mutex> lock(g_known_mu);
    const int i = g_known_used < kKnown ? g_known_used++ : (g_known_next++ % kKnown);
    g_known[i] = Known{ctx, *addr};
  }
  return cudaSuccess;
}

int64_t align256(int64_t x) { return (x + 255) / 256 * 256; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" pa_status pa_decode_splitkv_noalloc(
    void *out, const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int32_t num_pages, float scale,
    int32_t pages_per_split, pa_dtype dtype, int32_t *dev_err, pa_stream_t stream) {
  // pa_decode_splitkv's checks first, in its order, so that both entry points
  // give the same status for the same arguments
  pa_status st = pa::check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (pages_per_split <= 0) return PA_ERR_INVALID_ARG;
  const int32_t splits = pa_num_splits(max_blocks_per_seq, pages_per_split);
  if (static_cast<int64_t>(splits) * num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  // then the array's limit, and the output (checked here so that a bad `out`
  // is refused before the split read is launched)
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads * splits;
  const int64_t out_bytes = align256(rows * head_dim * static_cast<int64_t>(sizeof(float)));
  const int64_t lse_bytes = align256(rows * static_cast<int64_t>(sizeof(float)));
  if (out_bytes + lse_bytes > static_cast<int64_t>(PA_NOALLOC_SCRATCH_BYTES))
    return PA_ERR_UNSUPPORTED;  // partials would not fit the fixed array
  if (out == nullptr || !aligned16(out)) return PA_ERR_INVALID_ARG;

  unsigned char *base = nullptr;
  if (partials_address(&base) != cudaSuccess) return PA_ERR_CUDA;
  float *partial_out = reinterpret_cast<float *>(base);
  float *partial_lse = reinterpret_cast<float *>(base + out_bytes);

  st = pa_decode_splitkv(partial_out, partial_lse, q, k_pool, v_pool, block_table,
                         max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                         head_dim, block_size, num_pages, scale, pages_per_split, splits, dtype,
                         dev_err, stream);
  if (st != PA_OK) return st;
  return pa_merge(out, partial_out, partial_lse, num_seqs, num_q_heads, splits, head_dim, dtype,
                  stream);
}
