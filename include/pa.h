/*
 * pa.h - C ABI of the GB300 paged KV-cache decode-attention library (libpa.so).
 *
 * The cache is a fixed pool of pages.  A page holds block_size consecutive
 * tokens of one sequence; a sequence's block table lists its pages in order,
 * so token p of sequence b lives at slot p % block_size of page
 * block_table[b][p / block_size] ("Three Attention Kernels", section
 * "3. Paged KV-cache attention": the page comes from the block table, the
 * row from the offset inside the page).
 *
 * Memory layouts (row-major, contiguous, no padding):
 *   q, out        [num_seqs][num_q_heads][head_dim]                      dtype
 *   k_pool,v_pool [num_pages][block_size][num_kv_heads][head_dim]        dtype
 *   k_new,v_new   [num_tokens][num_kv_heads][head_dim]                   dtype
 *   block_table   [num_seqs][max_blocks_per_seq]                         int32
 *   seq_lens      [num_seqs]                                             int32
 *   partial_out   [num_seqs][num_q_heads][max_splits][head_dim]          float
 *   partial_lse   [num_seqs][num_q_heads][max_splits]                    float
 * Query head h reads kv head h / (num_q_heads / num_kv_heads) (grouped-query
 * attention with contiguous groups).
 *
 * Ownership: every pointer is device memory owned by the caller.  The
 * library allocates no memory and launches its kernels asynchronously on the
 * caller's stream; the call returns once the launch is queued.  Between
 * calls it keeps only host-side facts looked up once per CUDA context (each
 * kernel's shared-memory setting, the SM count and occupancy, recently
 * encoded tensor maps of the pools, the device address of the array behind
 * pa_decode_splitkv_noalloc) and that fixed array itself.  Cached facts are
 * keyed by the driver's context id, which is unique for the life of the
 * process, so they stay correct across a device reset or a change of
 * context.
 *
 * Errors: argument checks run on the host before any launch and return
 * PA_ERR_INVALID_ARG (a null or misaligned pointer, a negative or
 * inconsistent size) or PA_ERR_UNSUPPORTED (a valid shape the kernels do
 * not cover); nothing is launched then.  PA_ERR_CUDA means the launch
 * itself failed.  Values that live on the device (block-table entries,
 * sequence lengths, positions, sequence ids) are checked by the kernels:
 * an out-of-range value makes the kernel skip the memory access, write
 * zeros to the outputs it owns (lse -inf for split partials) and record the
 * first such error code in *dev_err (atomic compare-and-swap from 0; a null
 * dev_err only skips the recording).  No kernel traps or waits on another.
 *
 * Supported: dtype f32, f16 or bf16, the same for q, the pools, k_new/v_new
 * and out; head_dim * element size a multiple of 16 bytes and head_dim at
 * most 256; num_q_heads a multiple of num_kv_heads with at most 8 query
 * heads per kv head (16 for f16/bf16 with head_dim 32, 48, 64, 96, 128 or
 * 256); block_size a power of two from 1 to 1024; num_seqs at
 * most 65535.  All data pointers 16-byte aligned.
 */
#ifndef PA_H_
#define PA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st *pa_stream_t;

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,
  PA_ERR_UNSUPPORTED = 2,
  PA_ERR_CUDA = 3
} pa_status;

typedef enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2 } pa_dtype;

/* Codes a kernel records in *dev_err. */
enum {
  PA_DEV_OK = 0,
  PA_DEV_BAD_PAGE = 1,     /* block-table entry outside [0, num_pages) */
  PA_DEV_BAD_POSITION = 2, /* append position outside [0, max_blocks_per_seq * block_size) */
  PA_DEV_BAD_SEQ_LEN = 3,  /* seq_len outside [0, max_blocks_per_seq * block_size] */
  PA_DEV_BAD_SEQ_ID = 4,   /* append seq id outside [0, num_seqs) */
  PA_DEV_BAD_ITEM = 5,     /* work item with a bad sequence, range or slot */
  PA_DEV_TIMEOUT = 6       /* a bounded wait for the tensor cores ran out (output zeroed) */
};

/* Human-readable name of a status code (static string). */
const char *pa_status_string(pa_status status);

/* Library version string (static). */
const char *pa_version(void);

/* Splits per sequence for a split-KV read: ceil(max_blocks_per_seq /
 * pages_per_split), or 0 if either argument is not positive.  Sizes
 * partial_out and partial_lse. */
int32_t pa_num_splits(int32_t max_blocks_per_seq, int32_t pages_per_split);

/*
 * pa_cache_append - write new tokens' K and V into their page slots.
 *
 * nanoserve "Day 20: the number the Triton kernel has to beat", section
 * "What I learned": the cache write grows the block table and scatters the
 * K/V.  The table is grown by the caller (page allocation is host-side);
 * this call is the scatter.  Token i belongs to sequence seq_ids[i] (token
 * i belongs to sequence i when seq_ids is NULL) and is stored at position
 * positions[i]: k_new[i] (num_kv_heads * head_dim elements) is copied to
 * k_pool[block_table[seq][pos / block_size]][pos % block_size], likewise V.
 * A pure byte copy (no conversion): bit-exact, every other pool byte keeps
 * its value.  Two tokens of one call that name the same slot race.
 * num_tokens == 0 is a no-op.  num_seqs is the number of block-table rows.
 */
pa_status pa_cache_append(const void *k_new, const void *v_new, void *k_pool,
                          void *v_pool, const int32_t *block_table,
                          int32_t num_seqs, int32_t max_blocks_per_seq,
                          const int32_t *seq_ids, const int32_t *positions,
                          int32_t num_tokens, int32_t num_pages,
                          int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, pa_dtype dtype, int32_t *dev_err,
                          pa_stream_t stream);

/*
 * pa_decode - one decode step of attention over the paged cache.
 *
 * For every sequence b and query head h (kv head g = h / group):
 *   out[b][h] = softmax_t(scale * q[b][h] . K_b[t][g]) @ V_b[t][g],
 *   t = 0 .. seq_lens[b]-1,
 * where K_b[t] is read through the block table.  This is attention
 * softmax(Q K^T / sqrt(d)) V ("Three Attention Kernels", section "What is
 * attention, really?") at decode (one query per sequence), computed in one
 * streaming pass with an online softmax (a running max and sum, the score
 * row never stored) as nanoserve "Day 23: the real triton.jit
 * paged-attention kernel" streams its tiles.  seq_lens[b] counts every
 * attended token, including one appended this step.  A length of 0 gives
 * out = 0.  Accumulation is in fp32; out is rounded to dtype
 * (round-to-nearest-even).
 *
 * One CTA reads one (sequence, kv head) in launch order and sees only the
 * lengths on the device.  For a ragged batch whose lengths the caller has on
 * the host, the entry point is pa_plan_work + pa_decode_work + pa_merge:
 * near-equal work items, longest first, so that short sequences fill the end
 * of the grid (on 256 sequences of 16-8192 tokens, head_dim 128, it reads
 * in 650 us what this call reads in 708 us on a GB300).
 */
pa_status pa_decode(void *out, const void *q, const void *k_pool,
                    const void *v_pool, const int32_t *block_table,
                    int32_t max_blocks_per_seq, const int32_t *seq_lens,
                    int32_t num_seqs, int32_t num_q_heads,
                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                    int32_t num_pages, float scale, pa_dtype dtype,
                    int32_t *dev_err, pa_stream_t stream);

/*
 * pa_decode_splitkv - the same read, split along the history.
 *
 * "Three Attention Kernels", section "2. Split-KV flash-decoding": each
 * split reduces its own slice of K/V to a partial output and a log-sum-exp,
 * and a final cross-split combine (pa_merge) gives the output.  Here a split
 * is a fixed run of pages_per_split pages: split s of sequence b covers
 * tokens [s * pages_per_split * block_size, min(seq_lens[b], (s+1) *
 * pages_per_split * block_size)).  For every split it writes
 *   partial_out[b][h][s] = softmax-weighted V over the split (fp32),
 *   partial_lse[b][h][s] = log(sum_t exp(scale * q . k_t)) over the split,
 * and for a split with no tokens partial_out = 0, partial_lse = -inf.
 * max_splits must be at least pa_num_splits(max_blocks_per_seq,
 * pages_per_split); it is the split stride of the partial arrays.
 */
pa_status pa_decode_splitkv(float *partial_out, float *partial_lse,
                            const void *q, const void *k_pool,
                            const void *v_pool, const int32_t *block_table,
                            int32_t max_blocks_per_seq, const int32_t *seq_lens,
                            int32_t num_seqs, int32_t num_q_heads,
                            int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_pages, float scale,
                            int32_t pages_per_split, int32_t max_splits,
                            pa_dtype dtype, int32_t *dev_err,
                            pa_stream_t stream);

/*
 * pa_merge - combine split partials into the output.
 *
 * "Three Attention Kernels", section "2. Split-KV flash-decoding", the
 * cross-SM combine: for every (b, h), M = max_s partial_lse[b][h][s],
 * w_s = exp(partial_lse[b][h][s] - M), and
 *   out[b][h] = sum_s w_s * partial_out[b][h][s] / sum_s w_s,
 * rounded to dtype.  A row whose splits are all empty (every lse -inf)
 * gives 0.  fp32 arithmetic.  head_dim must be a multiple of 4 (every
 * supported read produces one) and partial_out 16-byte aligned.
 */
pa_status pa_merge(void *out, const float *partial_out,
                   const float *partial_lse, int32_t num_seqs,
                   int32_t num_q_heads, int32_t max_splits, int32_t head_dim,
                   pa_dtype dtype, pa_stream_t stream);

/*
 * pa_plan_work - host-side work plan for a ragged batch (no device access).
 *
 * "Three Attention Kernels" ("Key Tradeoffs") finds that more splits is not
 * monotonically better, and the explainer page on kernels (FlashInfer,
 * "Technical Details") plans ragged batches on the host every step.  Given
 * the host copy of the lengths, this cuts every sequence into near-equal
 * token ranges ("items") of at least min_pages_per_item pages, sized so
 * that items * num_kv_heads is about target_ctas (a multiple of the SM
 * count is a good target).  A sequence shorter than one item is one item;
 * a sequence of length 0 is one empty item.  Items are ordered longest
 * first.  Each item is four int32: sequence, first token, end token
 * (exclusive), and slot | (items of that sequence << 16), slot being the
 * item's index within its sequence.  Writes at most max_items items to
 * `items` (host memory, [max_items][4]) and the largest per-sequence item
 * count to *max_slots.  Returns the number of items, or -1 for bad
 * arguments, too small a buffer (num_seqs + total pages / min pages
 * always suffices) or a sequence that would need more than 32767 items
 * (the slot field's 15 bits); the buffer is left unwritten then.
 */
int32_t pa_plan_work(const int32_t *seq_lens, int32_t num_seqs, int32_t num_kv_heads,
                     int32_t block_size, int32_t target_ctas, int32_t min_pages_per_item,
                     int32_t *items, int32_t max_items, int32_t *max_slots);

/*
 * pa_decode_work - the split read over a planned work list.
 *
 * Runs one CTA per (item, kv head) of `items` (device memory, the
 * [num_items][4] records of pa_plan_work, 16-byte aligned) and writes, for
 * every item of sequence b with slot j, partial_out[b][h][j] and
 * partial_lse[b][h][j] exactly as pa_decode_splitkv writes a split.  The
 * last item of a sequence also sets partial_lse to -inf for its unused
 * slots (up to max_slots; their partial_out is left as it is).  pa_merge
 * with max_splits = max_slots then gives the output.  Every sequence must
 * have its slots 0 .. count-1 covered exactly once, as pa_plan_work
 * produces; a malformed item records PA_DEV_BAD_ITEM and its CTA writes
 * nothing.  f16/bf16 with the tensor-core head dims only.
 */
pa_status pa_decode_work(float *partial_out, float *partial_lse, const int32_t *items,
                         int32_t num_items, int32_t max_slots, const void *q,
                         const void *k_pool, const void *v_pool,
                         const int32_t *block_table, int32_t max_blocks_per_seq,
                         const int32_t *seq_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                         int32_t num_pages, float scale, pa_dtype dtype, int32_t *dev_err,
                         pa_stream_t stream);

/*
 * pa_decode_chunk - causal read of a chunk of queries per sequence.
 *
 * nanoserve "Day 23: the real triton.jit paged-attention kernel": every
 * query position i of a chunk is its own program, offset by the tokens
 * already in the cache (past).  Each sequence b brings chunk_len queries
 * whose K/V are already appended; seq_lens[b] counts the history and the
 * chunk, so past = seq_lens[b] - chunk_len.  Query i sits at position
 * past + i and attends to tokens 0 .. past + i:
 *   out[b][i][h] = softmax_{t <= past+i}(scale * q[b][i][h] . K_b[t][g]) @ V_b[t][g].
 * A query at a negative position (chunk_len > seq_lens[b]) sees nothing and
 * its output is 0.  q and out are [num_seqs][chunk_len][num_q_heads][head_dim].
 * chunk_len == 1 is a single-query read; a prompt's prefill is the chunk
 * with chunk_len == seq_lens[b].  f16/bf16 only, head_dim 32, 48, 64, 96 or
 * 128 (otherwise PA_ERR_UNSUPPORTED); fp32 accumulation and softmax, the
 * probabilities rounded to the cache dtype for the P.V product.  Chunks of
 * one query, or of up to 16 (query, head) columns per kv head at head_dim 64
 * (8 at head_dim 128), run on the single-query read's kernel with a causal
 * limit per column; larger ones at head_dim 64 and 128 on the tcgen05
 * tensor cores (two Q tiles per CTA from 256 rows, except head_dim-64 chunks
 * longer than an eighth of the table's capacity); the other head dims on the
 * mma.sync chunk kernel.
 * chunk_len * (num_q_heads / num_kv_heads) above 2^30 (query, head) rows
 * per kv head returns PA_ERR_UNSUPPORTED.
 *
 * The tcgen05 reads wait on mbarriers with a bound (about a second per wait);
 * a wait that runs out records PA_DEV_TIMEOUT in *dev_err, the affected
 * outputs are zeroed and the context stays usable (pa_test_set_withhold_tiles
 * makes that happen on purpose).
 */
pa_status pa_decode_chunk(void *out, const void *q, const void *k_pool,
                          const void *v_pool, const int32_t *block_table,
                          int32_t max_blocks_per_seq, const int32_t *seq_lens,
                          int32_t num_seqs, int32_t chunk_len, int32_t num_q_heads,
                          int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                          int32_t num_pages, float scale, pa_dtype dtype,
                          int32_t *dev_err, pa_stream_t stream);

/*
 * pa_decode_chunk_splitkv - the chunked read split into fixed page runs.
 *
 * "Three Attention Kernels", section "2. Split-KV flash-decoding", applied
 * to pa_decode_chunk: split s of sequence b covers pages
 * [s * pages_per_split, min((s+1) * pages_per_split, ceil(seq_lens[b] / block_size)))
 * as in pa_decode_splitkv, and query i keeps the tokens of that run at or
 * before its position past + i.  For every (b, i, h, s) it writes
 *   partial_out[b][i][h][s][:] = softmax-weighted V over those tokens (fp32),
 *   partial_lse[b][i][h][s]    = log(sum of exp(scale * q . k) over them),
 * and 0 / -inf where a query sees no token of the run.  pa_merge with
 * num_seqs * chunk_len as its sequence count combines them into the output
 * of pa_decode_chunk.  This is the form for long histories, where one CTA
 * per (sequence, kv head) would leave most of the GPU idle.
 *
 * partial_out [num_seqs][chunk_len][num_q_heads][max_splits][head_dim] and
 * partial_lse [num_seqs][chunk_len][num_q_heads][max_splits] are
 * caller-owned device float arrays (partial_out 16-byte aligned);
 * max_splits >= pa_num_splits(max_blocks_per_seq, pages_per_split) and at
 * most 65535; splits past a sequence's length are written as empty.  Other
 * arguments, errors and supported shapes are those of pa_decode_chunk.
 */
pa_status pa_decode_chunk_splitkv(float *partial_out, float *partial_lse, const void *q,
                                  const void *k_pool, const void *v_pool,
                                  const int32_t *block_table, int32_t max_blocks_per_seq,
                                  const int32_t *seq_lens, int32_t num_seqs, int32_t chunk_len,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_pages, float scale,
                                  int32_t pages_per_split, int32_t max_splits, pa_dtype dtype,
                                  int32_t *dev_err, pa_stream_t stream);

/*
 * pa_test_set_withhold_tiles - test hook for the bounded waits (not for
 * production use).  While on (nonzero), the warp-specialized tcgen05 chunk
 * read (256 or more (query, head) rows per kv head) loads no key tile: its
 * waits run out after about a second each, and the call records
 * PA_DEV_TIMEOUT with zeroed outputs, with no copy or MMA in flight.  Off by
 * default; process-wide; affects launches issued while it is on.
 */
void pa_test_set_withhold_tiles(int32_t on);

/* Size of the library-owned partials array behind pa_decode_splitkv_noalloc. */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

/*
 * pa_decode_splitkv_noalloc - split-KV read and merge without caller scratch.
 *
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory, so cannot pass pa_decode_splitkv the space
 * for its partial results.  Examples are a plugin whose host framework owns
 * every device allocation and hands it only inputs and outputs, or a serving
 * loop that must not call cudaMalloc/cudaFree because they may synchronize
 * the device.  It computes what pa_decode_splitkv followed by pa_merge
 * computes: out[b][h] for every sequence and query head, with
 * splits = pa_num_splits(max_blocks_per_seq, pages_per_split).  The partials
 * live in an array of PA_NOALLOC_SCRATCH_BYTES that the library places in
 * device memory on every GPU that loads it, held until the process exits.
 * The call allocates nothing.
 *
 * Limit: the partials take num_seqs * num_q_heads * splits * (head_dim + 1)
 * floats (each part rounded up to 256 bytes).  A call that needs more than
 * PA_NOALLOC_SCRATCH_BYTES returns PA_ERR_UNSUPPORTED and launches nothing.
 * Arguments are checked first as in pa_decode_splitkv (same status for the
 * same arguments), then the limit, then out (non-null, 16-byte aligned).
 *
 * The array's device address belongs to the CUDA context the library's
 * module was loaded into.  The first call in a context (the first on a
 * device, and the first after a device reset or in another context) looks it
 * up with cudaGetSymbolAddress, with that context current; later calls in
 * the same context reuse it.  Make that first call before any stream
 * capture.  Call it with the device that owns the stream and the data
 * current.  Every call on a device shares the one array.  Nothing depends on
 * what an earlier call left there, but calls whose kernels overlap on the GPU
 * (different streams, different host threads) race on it.
 */
pa_status pa_decode_splitkv_noalloc(void *out, const void *q, const void *k_pool,
                                    const void *v_pool, const int32_t *block_table,
                                    int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t num_pages, float scale,
                                    int32_t pages_per_split, pa_dtype dtype,
                                    int32_t *dev_err, pa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
