// Host planning of mla_decode_noalloc into fixed-capacity arrays (no heap),
// and the layout of the library's fixed device scratch. Plain C++ with no CUDA
// call, so the host tests can check the plan on their own.
#pragma once

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "internal.h"

namespace mla {
namespace noalloc {

// ---- fixed limits of the scratch (16 MiB on every device that loads the library)
constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxBatch = 1024;    // sequences per call
constexpr int kMaxCtas = 1024;     // persistent CTAs (one per SM)
constexpr int kMaxItems = kMaxBatch + kMaxCtas;
constexpr int kMaxReduce = kMaxBatch;
constexpr int kMaxSlots = 500;     // partial (O, LSE) slots: 500 x 32 KB

constexpr size_t kItemsOff = 0;
constexpr size_t kIndptrOff = kItemsOff + sizeof(WorkItem) * kMaxItems;
constexpr size_t kReduceOff = kIndptrOff + 8192;
constexpr size_t kZeroOff = kReduceOff + sizeof(ReduceEntry) * kMaxReduce;
constexpr size_t kLseOff = kZeroOff + 2048;
constexpr size_t kPartOff = (kLseOff + sizeof(float) * kMaxSlots * kHeads + 255) / 256 * 256;
constexpr size_t kEnd = kPartOff + sizeof(float) * (size_t)kMaxSlots * kHeads * kVDim;
static_assert(sizeof(int32_t) * (kMaxCtas + 1) <= 8192, "indptr region");
static_assert(kEnd <= kScratchBytes, "scratch layout exceeds the array");
static_assert(kZeroOff % 256 == 0 && kLseOff % 256 == 0 && kIndptrOff % 256 == 0, "alignment");

// Work list in fixed-capacity arrays (no heap): the same split as the
// regular planner with its default options (64-row granules balanced across
// CTAs, chunks of at least 64 rows, one CTA per SM), without its cost per item.
struct FixedPlan {
  WorkItem items[kMaxItems];
  int32_t indptr[kMaxCtas + 1];
  ReduceEntry reduce[kMaxReduce];
  int64_t cuts[kMaxCtas + 1];
  int n_items, n_ctas, n_reduce, n_slots;
};

// Returns MLA_OK, MLA_ERR_INDPTR, or MLA_ERR_NOALLOC_LIMIT when a fixed capacity is exceeded.
inline int plan_fixed(int batch, const int32_t* ip, int num_sms, FixedPlan* fp) {
  constexpr int64_t G = 64, kMinRows = 64;
  if (ip[0] != 0) return MLA_ERR_INDPTR;
  int64_t total = 0;
  for (int b = 0; b < batch; ++b) {
    if (ip[b + 1] < ip[b]) return MLA_ERR_INDPTR;
    total += (int64_t)ip[b + 1] - ip[b];
  }
  // granules of G rows per sequence (no prefix-sum array: the cut loop below
  // walks the sequences forward once instead)
  int64_t U = 0;
  for (int b = 0; b < batch; ++b) U += ((int64_t)ip[b + 1] - ip[b] + G - 1) / G;
  const int64_t max_ctas = std::min<int64_t>(num_sms, kMaxCtas);
  int64_t target = U > 0 ? (U + max_ctas - 1) / max_ctas : 1;
  target = std::max<int64_t>(target, (kMinRows + G - 1) / G);
  const int64_t n = U > 0 ? std::min<int64_t>(max_ctas, (U + target - 1) / target) : 1;
  fp->cuts[0] = 0;
  fp->cuts[n] = total;
  int b = 0;
  int64_t gb = 0;  // granules before sequence b
  for (int64_t k = 1; k < n; ++k) {
    const int64_t g = U * k / n;  // increasing in k: the scan over sequences only moves forward
    while (b < batch - 1 && gb + ((int64_t)ip[b + 1] - ip[b] + G - 1) / G <= g) {
      gb += ((int64_t)ip[b + 1] - ip[b] + G - 1) / G;
      ++b;
    }
    const int64_t S = ip[b], L = (int64_t)ip[b + 1] - S;
    fp->cuts[k] = S + std::min<int64_t>((g - gb) * G, L);
  }
  // keep only non-empty ranges: range c = [cuts[c], cuts[c+1])
  int64_t m = 0;
  for (int64_t k = 0; k < n; ++k)
    if (fp->cuts[k + 1] > fp->cuts[k]) fp->cuts[++m] = fp->cuts[k + 1];
  if (m == 0) m = 1;  // no rows at all: one CTA writes the zero outputs
  fp->n_ctas = (int)m;
  for (int c = 0; c <= fp->n_ctas; ++c) fp->indptr[c] = 0;
  int n_items = 0, cta = 0;
  for (int b = 0; b < batch; ++b) {
    const int64_t S = ip[b], E = ip[b + 1];
    while (cta < fp->n_ctas - 1 && fp->cuts[cta + 1] <= S) ++cta;
    if (S == E) {
      if (n_items >= kMaxItems) return MLA_ERR_NOALLOC_LIMIT;
      fp->items[n_items++] = WorkItem{b, 0, 0, -1, 0, b, 0, 0};
      fp->indptr[cta + 1]++;
      continue;
    }
    while (true) {
      const int64_t a = std::max(S, fp->cuts[cta]), e = std::min(E, fp->cuts[cta + 1]);
      if (e > a) {
        if (n_items >= kMaxItems) return MLA_ERR_NOALLOC_LIMIT;
        fp->items[n_items++] = WorkItem{b, (int32_t)(a - S), (int32_t)(e - S), -1, (int32_t)(E - S), b, 0, 0};
        fp->indptr[cta + 1]++;
      }
      if (E <= fp->cuts[cta + 1] || cta == fp->n_ctas - 1) break;
      ++cta;
    }
  }
  for (int c = 0; c < fp->n_ctas; ++c) fp->indptr[c + 1] += fp->indptr[c];
  int slot = 0, n_reduce = 0;
  for (int i = 0; i < n_items;) {
    int j = i + 1;
    while (j < n_items && fp->items[j].b == fp->items[i].b) ++j;
    if (j - i > 1) {
      if (n_reduce >= kMaxReduce || slot + (j - i) > kMaxSlots) return MLA_ERR_NOALLOC_LIMIT;
      fp->reduce[n_reduce++] = ReduceEntry{fp->items[i].b, slot, j - i, 0};
      for (int k = i; k < j; ++k) fp->items[k].slot = slot++;
    }
    i = j;
  }
  fp->n_items = n_items;
  fp->n_reduce = n_reduce;
  fp->n_slots = slot;
  return MLA_OK;
}

}  // namespace noalloc
}  // namespace mla
