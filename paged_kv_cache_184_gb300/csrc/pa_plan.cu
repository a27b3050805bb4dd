// Host-side work planning for ragged batches (pa_plan_work).
//
// The split-KV read of "Three Attention Kernels" (section "2. Split-KV
// flash-decoding") uses one split count for the whole batch, and its
// "Key Tradeoffs" section finds that more splits is not monotonically
// better.  A ragged serving batch wants something else: long sequences
// split, short ones not, and the pieces sized so that the whole grid keeps
// every SM busy to the end.  The explainer page (FlashInfer, "Technical
// Details") describes exactly this as per-step planning on the host while
// the GPU computes.  This file is that planner: plain host code, run on the
// host copy of the lengths, producing a work list for pa_decode_work.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "pa_internal.h"

extern "C" int32_t pa_plan_work(const int32_t *seq_lens, int32_t num_seqs, int32_t num_kv_heads,
                                int32_t block_size, int32_t target_ctas,
                                int32_t min_pages_per_item, int32_t *items, int32_t max_items,
                                int32_t *max_slots) {
  if (seq_lens == nullptr || items == nullptr || max_slots == nullptr || num_seqs <= 0 ||
      num_kv_heads <= 0 || block_size <= 0 || target_ctas <= 0 || min_pages_per_item <= 0 ||
      max_items <= 0)
    return -1;
  // pages of every sequence, and their total
  std::vector<int64_t> pages(num_seqs);
  int64_t total = 0;
  for (int32_t b = 0; b < num_seqs; ++b) {
    if (seq_lens[b] < 0) return -1;
    pages[b] = (static_cast<int64_t>(seq_lens[b]) + block_size - 1) / block_size;
    total += pages[b];
  }
  // item size: the pages that give about target_ctas CTAs (each item runs on
  // num_kv_heads CTAs), never fewer than min_pages_per_item
  const int64_t target_items = std::max<int64_t>(1, target_ctas / num_kv_heads);
  const int64_t item_pages =
      std::max<int64_t>(min_pages_per_item, (total + target_items - 1) / target_items);

  struct Item {
    int32_t seq, begin, end, slot, count;
  };
  std::vector<Item> list;
  int32_t slots = 1;
  for (int32_t b = 0; b < num_seqs; ++b) {
    // as many items as fit whole: each at least item_pages, below 2 * item_pages
    const int64_t n = std::max<int64_t>(1, pages[b] / item_pages);
    if (n > 32767) return -1;  // the slot count must fit 15 bits of the item record
    // refuse a plan that outgrows the caller's buffer before building it
    if (static_cast<int64_t>(list.size()) + n > max_items) return -1;
    slots = std::max<int32_t>(slots, static_cast<int32_t>(n));
    // n near-equal page runs covering the sequence in order
    for (int64_t j = 0; j < n; ++j) {
      const int64_t p0 = pages[b] * j / n, p1 = pages[b] * (j + 1) / n;
      const int64_t t0 = std::min<int64_t>(seq_lens[b], p0 * block_size);
      const int64_t t1 = std::min<int64_t>(seq_lens[b], p1 * block_size);
      list.push_back({b, static_cast<int32_t>(t0), static_cast<int32_t>(t1),
                      static_cast<int32_t>(j), static_cast<int32_t>(n)});
    }
  }
  // longest first, so the shortest items fill the end of the grid
  std::stable_sort(list.begin(), list.end(), [](const Item &x, const Item &y) {
    return (x.end - x.begin) > (y.end - y.begin);
  });
  for (size_t i = 0; i < list.size(); ++i) {
    items[4 * i + 0] = list[i].seq;
    items[4 * i + 1] = list[i].begin;
    items[4 * i + 2] = list[i].end;
    items[4 * i + 3] = list[i].slot | (list[i].count << 16);
  }
  *max_slots = slots;
  return static_cast<int32_t>(list.size());
}
