// C ABI of libpa.so: argument validation and launch.
//
// Every integer the kernels turn into an address (strides, the grid, the
// split count, the block-size shift) is computed and checked here on the
// host, in plain code that runs without a GPU, as nanoserve "Day 23: the
// real triton.jit paged-attention kernel" keeps its index math outside the
// kernel.  Values that only exist on the device (block-table entries,
// lengths, positions) are checked by the kernels themselves.
#include <cmath>
#include <cstdint>

#include "pa_internal.h"

namespace {

constexpr int32_t kMaxHeadDim = 256;
constexpr int32_t kMaxGroupSimt = 8;   // CUDA-core read
constexpr int32_t kMaxGroupMma = 16;   // tensor-core read
constexpr int32_t kMaxBlockSize = 1024;
constexpr int32_t kMaxSeqs = 65535;  // grid.y
// (query, head) rows per kv head of a chunk: an int in the kernels, with room for rounding up
constexpr int64_t kMaxChunkRows = int64_t{1} << 30;

int elem_size(pa_dtype dt) {
  switch (dt) {
    case PA_F32: return 4;
    case PA_F16: return 2;
    case PA_BF16: return 2;
  }
  return 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int log2_exact(int32_t x) {  // -1 unless x is a power of two
  if (x <= 0 || (x & (x - 1)) != 0) return -1;
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

}  // namespace

// Checks shared by the reads: shapes, dtype, head dim, group, block size.
pa_status pa::check_read_shape(int32_t max_blocks, int32_t num_seqs, int32_t hq, int32_t hkv,
                           int32_t d, int32_t block_size, int32_t num_pages, float scale,
                           pa_dtype dtype) {
  if (max_blocks <= 0 || num_seqs < 0 || hq <= 0 || hkv <= 0 || d <= 0 || num_pages <= 0)
    return PA_ERR_INVALID_ARG;
  if (hq % hkv != 0) return PA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PA_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  if (es == 0) return PA_ERR_INVALID_ARG;
  if (log2_exact(block_size) < 0) return PA_ERR_INVALID_ARG;
  if (block_size > kMaxBlockSize) return PA_ERR_UNSUPPORTED;
  if ((static_cast<int64_t>(d) * es) % 16 != 0 || d > kMaxHeadDim) return PA_ERR_UNSUPPORTED;
  const int group = hq / hkv;
  if (group > kMaxGroupMma) return PA_ERR_UNSUPPORTED;
  if (group > kMaxGroupSimt && !pa::mma_supports(dtype, d, group)) return PA_ERR_UNSUPPORTED;
  if (num_seqs > kMaxSeqs) return PA_ERR_UNSUPPORTED;
  // the largest element offset of a pool must fit the kernels' size_t math and
  // a page count times rows must fit the int64 row index (always true here)
  return PA_OK;
}

namespace {

using pa::check_read_shape;

pa::DecodeParams make_params(const void *q, const void *k_pool, const void *v_pool,
                             const int32_t *block_table, int32_t max_blocks,
                             const int32_t *seq_lens, int32_t num_seqs, int32_t hq, int32_t hkv,
                             int32_t d, int32_t block_size, int32_t num_pages, float scale,
                             int32_t *dev_err) {
  pa::DecodeParams p{};
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.dev_err = dev_err;
  p.num_seqs = num_seqs;
  p.num_q_heads = hq;
  p.num_kv_heads = hkv;
  p.head_dim = d;
  p.group = hq / hkv;
  p.max_blocks = max_blocks;
  p.block_size_log2 = log2_exact(block_size);
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.chunk_len = 1;
  p.head_group = p.group;
  return p;
}

pa_status launched(cudaError_t err) { return err == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

// f16/bf16 rows the tensor-core kernel covers go there, fp32 to its CUDA-core
// read, the rest (f16/bf16 at other head dims) to the general CUDA-core read.
cudaError_t launch_read(const pa::DecodeParams &p, pa_dtype dtype, cudaStream_t stream) {
  if (pa::mma_supports(dtype, p.head_dim, p.group)) return pa::launch_decode_mma(p, dtype, stream);
  if (dtype == PA_F32 && p.chunk_len == 1) return pa::launch_decode_f32(p, stream);
  return pa::launch_decode_simt(p, dtype, stream);
}

}  // namespace

extern "C" {

const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
  }
  return "PA_ERR_UNKNOWN";
}

const char *pa_version(void) { return "paged_kv_cache_184_gb300 0.1 (sm_103a)"; }

int32_t pa_num_splits(int32_t max_blocks_per_seq, int32_t pages_per_split) {
  if (max_blocks_per_seq <= 0 || pages_per_split <= 0) return 0;
  return static_cast<int32_t>((static_cast<int64_t>(max_blocks_per_seq) + pages_per_split - 1) /
                              pages_per_split);
}

pa_status pa_cache_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                          const int32_t *block_table, int32_t num_seqs,
                          int32_t max_blocks_per_seq, const int32_t *seq_ids,
                          const int32_t *positions, int32_t num_tokens, int32_t num_pages,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          pa_dtype dtype, int32_t *dev_err, pa_stream_t stream) {
  if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq <= 0 || num_pages <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  const int es = elem_size(dtype);
  if (es == 0 || log2_exact(block_size) < 0) return PA_ERR_INVALID_ARG;
  if (block_size > kMaxBlockSize) return PA_ERR_UNSUPPORTED;
  const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * es;
  if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (row_bytes / 16 > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (seq_ids == nullptr && num_tokens > num_seqs) return PA_ERR_INVALID_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!k_new || !v_new || !k_pool || !v_pool || !block_table || !positions)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  pa::AppendParams p{};
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_ids = seq_ids;
  p.positions = positions;
  p.dev_err = dev_err;
  p.num_seqs = num_seqs;
  p.max_blocks = max_blocks_per_seq;
  p.num_tokens = num_tokens;
  p.num_pages = num_pages;
  p.block_size_log2 = log2_exact(block_size);
  p.row_chunks = static_cast<int32_t>(row_bytes / 16);
  return launched(pa::launch_append(p, reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_decode(void *out, const void *q, const void *k_pool, const void *v_pool,
                    const int32_t *block_table, int32_t max_blocks_per_seq,
                    const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int32_t num_pages, float scale, pa_dtype dtype, int32_t *dev_err,
                    pa_stream_t stream) {
  pa_status st = check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                  head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  pa::DecodeParams p = make_params(q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens,
                                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                   num_pages, scale, dev_err);
  p.out = out;
  p.pages_per_split = 0;
  p.num_splits = 1;
  return launched(launch_read(p, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_splitkv(float *partial_out, float *partial_lse, const void *q,
                            const void *k_pool, const void *v_pool, const int32_t *block_table,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                            int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int32_t num_pages, float scale,
                            int32_t pages_per_split, int32_t max_splits, pa_dtype dtype,
                            int32_t *dev_err, pa_stream_t stream) {
  pa_status st = check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                  head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (pages_per_split <= 0) return PA_ERR_INVALID_ARG;
  const int32_t need = pa_num_splits(max_blocks_per_seq, pages_per_split);
  if (max_splits < need) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_splits) * num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!partial_out || !partial_lse || !q || !k_pool || !v_pool || !block_table || !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(partial_out))
    return PA_ERR_INVALID_ARG;
  pa::DecodeParams p = make_params(q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens,
                                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                   num_pages, scale, dev_err);
  p.partial_out = partial_out;
  p.partial_lse = partial_lse;
  p.pages_per_split = pages_per_split;
  p.num_splits = max_splits;
  return launched(launch_read(p, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_work(float *partial_out, float *partial_lse, const int32_t *items,
                         int32_t num_items, int32_t max_slots, const void *q, const void *k_pool,
                         const void *v_pool, const int32_t *block_table,
                         int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, int32_t num_pages, float scale, pa_dtype dtype,
                         int32_t *dev_err, pa_stream_t stream) {
  pa_status st = check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                  head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (!pa::mma_supports(dtype, head_dim, num_q_heads / num_kv_heads)) return PA_ERR_UNSUPPORTED;
  if (max_slots <= 0 || max_slots > 32767 || num_items < 0) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(num_items) * num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (num_items == 0) return PA_ERR_INVALID_ARG;  // every sequence needs an item
  if (!partial_out || !partial_lse || !items || !q || !k_pool || !v_pool || !block_table ||
      !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(items) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) ||
      !aligned16(partial_out))
    return PA_ERR_INVALID_ARG;
  pa::DecodeParams p = make_params(q, k_pool, v_pool, block_table, max_blocks_per_seq, seq_lens,
                                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                   num_pages, scale, dev_err);
  p.partial_out = partial_out;
  p.partial_lse = partial_lse;
  p.pages_per_split = 0;
  p.num_splits = max_slots;
  p.items = items;
  p.num_items = num_items;
  return launched(pa::launch_decode_items(p, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

// The chunk read for this many (query, head) rows per kv head.  From 256 rows
// (two full 128-row tiles) the warp-specialized tcgen05 read with two Q tiles per
// CTA, except at head_dim 64 when the chunk is more than an eighth of the table's
// capacity (a prefill, say): there the pipelined one-tile read, four CTAs per SM,
// measured faster (prefills of 8 x 4096 / 32 x 1024 / 64 x 512 tokens: 786 / 289
// / 213 us against 842 / 377 / 299), while on a short chunk of a long history the
// two Q tiles sharing each K/V load pay (128 queries at history 4096: 383 against
// 411 us).  Below 256 rows the pipelined read at head_dim 64 and 128 (every chunk
// that reaches here: the decode kernel takes up to 16 columns at 64, 8 at 128);
// mma.sync at the other head dims.
static cudaError_t launch_chunk_read(const pa::ChunkParams &p, pa_dtype dtype, int64_t rows,
                                     cudaStream_t s) {
  const int r = static_cast<int>(rows);
  const long long capacity = static_cast<long long>(p.max_blocks) << p.block_size_log2;
  const bool long_chunk = static_cast<long long>(p.chunk_len) * 8 > capacity;
  if (pa::chunk_tc_ws_supports(dtype, p.head_dim, r) && !(p.head_dim == 64 && long_chunk))
    return pa::launch_chunk_tc_ws(p, dtype, s);
  if (pa::chunk_tc_pipe_supports(dtype, p.head_dim, r))
    return pa::launch_chunk_tc_pipe(p, dtype, s);
  return pa::launch_chunk(p, dtype, s);
}

pa_status pa_decode_chunk(void *out, const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_table, int32_t max_blocks_per_seq,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t chunk_len,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_pages, float scale, pa_dtype dtype,
                          int32_t *dev_err, pa_stream_t stream) {
  if (chunk_len <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                  head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (!pa::chunk_supports(dtype, head_dim)) return PA_ERR_UNSUPPORTED;
  const int64_t rows = static_cast<int64_t>(chunk_len) * (num_q_heads / num_kv_heads);
  if (rows > kMaxChunkRows) return PA_ERR_UNSUPPORTED;
  const int64_t ctas = (rows + pa::chunk_rows_per_cta() - 1) / pa::chunk_rows_per_cta();
  if (ctas * num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_table || !seq_lens) return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int group = num_q_heads / num_kv_heads;
  // one query per sequence is the single-query read; up to 16 (query, head)
  // columns per kv head run on its tensor-core kernel with per-column limits
  if (chunk_len == 1 || pa::mma_chunk_supports(dtype, head_dim, static_cast<int>(rows))) {
    pa::DecodeParams dp = make_params(q, k_pool, v_pool, block_table, max_blocks_per_seq,
                                      seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      block_size, num_pages, scale, dev_err);
    dp.out = out;
    dp.pages_per_split = 0;
    dp.num_splits = 1;
    dp.chunk_len = chunk_len;
    dp.group = chunk_len * group;
    return launched(launch_read(dp, dtype, s));
  }
  pa::ChunkParams p{};
  p.out = out;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.dev_err = dev_err;
  p.num_seqs = num_seqs;
  p.chunk_len = chunk_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.group = num_q_heads / num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.block_size_log2 = log2_exact(block_size);
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  return launched(launch_chunk_read(p, dtype, rows, s));
}

pa_status pa_decode_chunk_splitkv(float *partial_out, float *partial_lse, const void *q,
                                  const void *k_pool, const void *v_pool,
                                  const int32_t *block_table, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, int32_t num_seqs, int32_t chunk_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_pages, float scale,
                                  int32_t pages_per_split, int32_t max_splits, pa_dtype dtype,
                                  int32_t *dev_err, pa_stream_t stream) {
  if (chunk_len <= 0 || pages_per_split <= 0) return PA_ERR_INVALID_ARG;
  pa_status st = check_read_shape(max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads,
                                  head_dim, block_size, num_pages, scale, dtype);
  if (st != PA_OK) return st;
  if (!pa::chunk_supports(dtype, head_dim)) return PA_ERR_UNSUPPORTED;
  const int32_t need = pa_num_splits(max_blocks_per_seq, pages_per_split);
  if (max_splits < need) return PA_ERR_INVALID_ARG;
  if (max_splits > 65535) return PA_ERR_UNSUPPORTED;  // the split is the grid's z index
  const int64_t rows = static_cast<int64_t>(chunk_len) * (num_q_heads / num_kv_heads);
  if (rows > kMaxChunkRows) return PA_ERR_UNSUPPORTED;
  const int64_t ctas = (rows + pa::chunk_rows_per_cta() - 1) / pa::chunk_rows_per_cta();
  if (ctas * num_kv_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!partial_out || !partial_lse || !q || !k_pool || !v_pool || !block_table || !seq_lens)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(partial_out))
    return PA_ERR_INVALID_ARG;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int group = num_q_heads / num_kv_heads;
  if (chunk_len == 1 || pa::mma_chunk_supports(dtype, head_dim, static_cast<int>(rows))) {
    pa::DecodeParams dp = make_params(q, k_pool, v_pool, block_table, max_blocks_per_seq,
                                      seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                      block_size, num_pages, scale, dev_err);
    dp.partial_out = partial_out;
    dp.partial_lse = partial_lse;
    dp.pages_per_split = pages_per_split;
    dp.num_splits = max_splits;
    dp.chunk_len = chunk_len;
    dp.group = chunk_len * group;
    return launched(launch_read(dp, dtype, s));
  }
  pa::ChunkParams p{};
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.dev_err = dev_err;
  p.partial_out = partial_out;
  p.partial_lse = partial_lse;
  p.pages_per_split = pages_per_split;
  p.num_splits = max_splits;
  p.num_seqs = num_seqs;
  p.chunk_len = chunk_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.group = num_q_heads / num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.block_size_log2 = log2_exact(block_size);
  p.num_pages = num_pages;
  p.scale_log2 = scale * 1.4426950408889634f;
  return launched(launch_chunk_read(p, dtype, rows, s));
}

pa_status pa_merge(void *out, const float *partial_out, const float *partial_lse,
                   int32_t num_seqs, int32_t num_q_heads, int32_t max_splits, int32_t head_dim,
                   pa_dtype dtype, pa_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_splits <= 0 || head_dim <= 0)
    return PA_ERR_INVALID_ARG;
  if (elem_size(dtype) == 0) return PA_ERR_INVALID_ARG;
  if (head_dim > kMaxHeadDim || head_dim % 4 != 0) return PA_ERR_UNSUPPORTED;
  const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads;
  if (rows > INT32_MAX / 4) return PA_ERR_UNSUPPORTED;
  if (rows == 0) return PA_OK;
  if (!out || !partial_out || !partial_lse) return PA_ERR_INVALID_ARG;
  if (!aligned16(partial_out)) return PA_ERR_INVALID_ARG;  // read as float4 rows
  pa::MergeParams p{};
  p.out = out;
  p.partial_out = partial_out;
  p.partial_lse = partial_lse;
  p.rows = static_cast<int32_t>(rows);
  p.num_splits = max_splits;
  p.head_dim = head_dim;
  return launched(pa::launch_merge(p, dtype, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
