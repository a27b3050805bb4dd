// Internal interface between the C-ABI layer (pa_api.cu) and the kernels.
// Every pointer is caller-owned device memory; every size was validated by
// the C-ABI layer before any launcher here is called.
#pragma once

#include <cuda.h>  // CUtensorMap
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pa.h"

namespace pa {

// Launch with programmatic stream serialization, so the kernel's launch and
// prologue overlap the tail of the previous kernel in the stream; the kernel
// must call pdl_wait() before touching memory the previous kernel writes.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Per-context host cache (pa_host.cu).  Each fact is looked up once per CUDA
// context (keyed by the driver's process-unique context id), so a launch
// repeats no runtime query; with no current context the query runs uncached.
uint64_t current_context_id();  // 0 when no context is current or it has no id
// cudaFuncSetAttribute(kern, MaxDynamicSharedMemorySize, smem), once per context.
cudaError_t set_max_smem(const void *kern, int smem);
// Streaming multiprocessors of the current device.
cudaError_t sm_count(int *sms);
// Resident CTAs per SM of `kern` at `threads` threads and `smem` dynamic shared
// bytes (also sets the kernel's shared-memory limit to smem).
cudaError_t blocks_per_sm(int *n, const void *kern, int threads, int smem);

// Shape checks shared by every read entry point (pa_api.cu): sizes, dtype,
// head dim, group and block size, before any pointer is looked at.
pa_status check_read_shape(int32_t max_blocks, int32_t num_seqs, int32_t hq, int32_t hkv,
                           int32_t d, int32_t block_size, int32_t num_pages, float scale,
                           pa_dtype dtype);

// Arguments of one paged read (pa_decode or pa_decode_splitkv).
struct DecodeParams {
  void *out;            // [B][Hq][D] dtype; unused by the split-KV read
  float *partial_out;   // [B][Hq][max_splits][D]; split-KV read only
  float *partial_lse;   // [B][Hq][max_splits];    split-KV read only
  const void *q;        // [B][Hq][D]
  const void *k_pool;   // [num_pages][block_size][Hkv][D]
  const void *v_pool;
  const int32_t *block_table;  // [B][max_blocks]
  const int32_t *seq_lens;     // [B]
  int32_t *dev_err;            // nullable
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim, group;
  int32_t max_blocks, block_size_log2, num_pages;
  int32_t pages_per_split;  // 0: one split spanning the whole sequence
  int32_t num_splits;       // splits per sequence, the partials' split stride (1 if unsplit)
  int32_t splits_per_cta;   // consecutive splits one CTA reads (tensor-core read; else 1)
  int32_t comb_heads;       // head slots per warp in the combine area (tensor-core read)
  const int32_t *items;     // work list [num_items][4] (pa_decode_work), else null
  int32_t num_items;
  float scale_log2;         // scale * log2(e): scores kept in base-2 units
  // Chunked read on this kernel (tensor-core read, chunk_len > 1): `group`
  // counts the CTA's columns, chunk_len * head_group (query, head) pairs, and
  // column c is query c / head_group, head c % head_group of the kv head;
  // q and out are [B][chunk_len][Hq][D], the partials [B][chunk_len][Hq][S][D].
  int32_t chunk_len;        // 1 for the single-query read
  int32_t head_group;       // query heads per kv head (Hq / Hkv)
};

// Arguments of the chunked multi-query read (pa_decode_chunk).
struct ChunkParams {
  void *out;                   // [B][chunk_len][Hq][D] (one-pass read)
  const void *q;               // [B][chunk_len][Hq][D]
  const void *k_pool, *v_pool;
  const int32_t *block_table, *seq_lens;
  int32_t *dev_err;
  // split read (partial_out non-null): blockIdx.z is the split, which covers
  // pages [z * pages_per_split, (z + 1) * pages_per_split) of the sequence
  float *partial_out;          // [B][chunk_len][Hq][num_splits][D]
  float *partial_lse;          // [B][chunk_len][Hq][num_splits]
  int32_t pages_per_split, num_splits;
  int32_t num_seqs, chunk_len, num_q_heads, num_kv_heads, head_dim, group;
  int32_t max_blocks, block_size_log2, num_pages;
  float scale_log2;
};

struct AppendParams {
  const void *k_new, *v_new;  // [T][Hkv][D]
  void *k_pool, *v_pool;
  const int32_t *block_table, *seq_ids, *positions;
  int32_t *dev_err;
  int32_t num_seqs, max_blocks, num_tokens, num_pages, block_size_log2;
  int32_t row_chunks;  // 16-byte chunks in one token row (Hkv * D * elem / 16)
};

struct MergeParams {
  void *out;
  const float *partial_out, *partial_lse;
  int32_t rows;  // B * Hq
  int32_t num_splits, head_dim;
};

// CUDA-core read for f16/bf16 at head dims outside the tensor-core list, groups of up to 8.
cudaError_t launch_decode_simt(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream);
// CUDA-core read for fp32 caches (pa_decode_f32.cu): groups of up to 8.
cudaError_t launch_decode_f32(const DecodeParams &p, cudaStream_t stream);
// Tensor-core read: f16/bf16, head_dim in {32, 48, 64, 96, 128, 256}, groups of up to 16.
bool mma_supports(pa_dtype dtype, int head_dim, int group);
// The chunked read of up to 16 (query, head) columns per kv head at head_dim
// 64, or 8 at head_dim 128, on the tensor-core decode kernel (f16/bf16).
bool mma_chunk_supports(pa_dtype dtype, int head_dim, int columns);
cudaError_t launch_decode_mma(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream);
// Tensor-core read over a planned work list (p.items), same shapes as above.
cudaError_t launch_decode_items(const DecodeParams &p, pa_dtype dtype, cudaStream_t stream);
// Chunked multi-query read: f16/bf16, head_dim in {32, 48, 64, 96, 128}.
bool chunk_supports(pa_dtype dtype, int head_dim);
int chunk_rows_per_cta();
cudaError_t launch_chunk(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream);

// warp-specialized tcgen05 chunk read (pa_chunk_tc_ws.cu): two 128-row Q tiles per CTA
bool chunk_tc_ws_supports(pa_dtype dtype, int head_dim, int rows);
cudaError_t launch_chunk_tc_ws(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream);
// pipelined tcgen05 chunk read (pa_chunk_tc_pipe.cu): one 128-row Q tile per CTA, S
// double-buffered, several CTAs per SM
bool chunk_tc_pipe_supports(pa_dtype dtype, int head_dim, int rows);
cudaError_t launch_chunk_tc_pipe(const ChunkParams &p, pa_dtype dtype, cudaStream_t stream);
// A 2D tensor map of a pool (token rows of Hkv * D elements, 128-byte swizzle) whose box
// is 64 elements by min(block_size, box_rows) rows, from a small cache of encoded maps
// (pa_chunk_tc_ws.cu); false when the driver's encoder is unavailable or refuses.
bool pool_tensor_map(CUtensorMap *map, const void *pool, pa_dtype dtype, const ChunkParams &p,
                     int box_rows);
// State of the time-out test hook (pa_test_set_withhold_tiles): nonzero makes the
// tcgen05 chunk reads' loaders announce no tile, so that their bounded waits run out.
int withhold_tiles();
cudaError_t launch_append(const AppendParams &p, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams &p, pa_dtype dtype, cudaStream_t stream);

}  // namespace pa
