// Host split-KV planner.
//
// The pages build a persistent-mode work list on the host side of every call
// shape and cache it (get_mla_metadata_info_v1 / get_mla_metadata_v1 in
// kernelbot amd-mixed-mla submission 598454 "v12", _get_or_compute_metadata;
// kv_granularity = max(page_size, 16) there). Their field layout belongs to a
// closed library and is not shown, so this planner defines its own: the rows
// of all sequences, laid end to end, are cut into one contiguous range per
// persistent CTA holding the same number of `granularity`-row granules (to
// within one). A sequence that lies inside one range is a single work item
// writing its final output; a sequence that straddles cuts becomes several
// items writing partial (O, LSE) slots that the reduce merges. Cuts fall on
// multiples of `granularity` rows from the sequence start, and no range is
// shorter than `min_rows_per_split` unless the whole problem is.
#include <algorithm>
#include <climits>
#include <cstdint>
#include <utility>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "internal.h"

namespace mla {

PlanOptions resolve_options(const mla_plan_options* o) {
  PlanOptions r;
  if (!o) return r;
  if (o->num_kv_slots > 0) r.num_kv_slots = o->num_kv_slots;
  if (o->min_rows_per_split > 0) r.min_rows_per_split = o->min_rows_per_split;
  if (o->granularity > 0) r.granularity = o->granularity;
  if (o->ctas_per_sm > 0) r.ctas_per_sm = o->ctas_per_sm;
  if (o->fp8_kernel == 1) r.fp8_kernel = 1;
  if (o->fp8_issuers == 1 || o->fp8_issuers == 2) r.fp8_issuers = o->fp8_issuers;
  if (o->item_cost_rows > 0) r.item_cost_rows = o->item_cost_rows;
  if (o->item_cost_rows < 0) r.item_cost_rows = 0;
  if (o->token_parallel < 0) r.token_parallel = false;
  if (o->token_pairs > 0) r.token_pairs = true;
  return r;
}

void free_host_plan(HostPlan* p) {
  std::free(p->items);
  std::free(p->work_indptr);
  std::free(p->reduce);
  p->items = nullptr;
  p->work_indptr = nullptr;
  p->reduce = nullptr;
}

namespace {

// The planner proper, on the sequences' token counts laid end to end:
// tok[b] is the first token of sequence b in that concatenation, tok[batch]
// the total; qo[b] is the first query row of sequence b, qo[batch] the number
// of query rows (single-token plans: qo[b] = b).
int plan_tokens(int batch, const std::vector<int64_t>& tok, const std::vector<int64_t>& qo, bool causal, int num_sms,
                const PlanOptions& opt, HostPlan* out) {
  const int64_t total = tok[(size_t)batch];
  out->total_rows = total;
  auto seq_len = [&](int b) { return tok[(size_t)b + 1] - tok[(size_t)b]; };
  auto n_queries = [&](int b) { return qo[(size_t)b + 1] - qo[(size_t)b]; };
  // KV tokens query token j of sequence b sees (its causal prefix, or all)
  auto visible = [&](int b, int64_t j) {
    const int64_t L = seq_len(b);
    const int64_t n = causal ? L - n_queries(b) + j + 1 : L;
    return std::min<int64_t>(std::max<int64_t>(n, 0), L);
  };

  // Work is counted in granules: sequence b is ceil(L_b / G) granules of G
  // rows (its last one may be shorter), each weighing the number of query
  // tokens that read it. Every item a range starts (one per query token of each
  // sequence piece it holds) adds a fixed cost of item_cost_rows rows: an item
  // boundary costs a CTA an epilogue, a query staging and a pipeline refill,
  // measured at about two tiles' time. Ranges are cut, on multiples of G rows
  // from each sequence's start, so that the largest range cost is as small as
  // the number of CTAs allows (binary search on that cost, filling greedily).
  // With one query token per sequence, no item cost and G equal to the
  // kernels' tile height, the ranges hold the same number of tiles to within
  // one. A range reads each of its KV rows from HBM once; the query tokens of
  // one sequence run back to back over the same rows.
  const int64_t G = opt.granularity;
  int64_t max_ctas = (int64_t)num_sms * opt.ctas_per_sm;
  const int64_t kUnit = 16;  // cost units per granule, so that an item cost below one granule still counts
  const int64_t item_cost = (int64_t)opt.item_cost_rows * kUnit / G;
  const int64_t min_granules = (opt.min_rows_per_split + G - 1) / G;
  std::vector<int64_t> ngran((size_t)batch, 0);
  for (int b = 0; b < batch; ++b) ngran[(size_t)b] = (seq_len(b) + G - 1) / G;
  // Token-parallel plans: when every sequence with KV rows has the same number Q > 1
  // of query tokens, the row ranges are planned for one token over max_ctas / Q
  // CTAs, and each range becomes Q CTAs, one per query token, side by side in the
  // grid. They read the same rows at the same time: the rows come from HBM once
  // and from L2 for the other tokens (a range processing its tokens back to back
  // re-reads them from HBM once the ranges outgrow L2).
  //
  // Token pairs (asked for by the option; a multi-token plan builds this list
  // beside the per-token one): when that Q is even, query tokens 2v and 2v+1 of a
  // sequence form one unit, processed in one pass over their rows by the fp8
  // tensor-core kernel. A pair item covers rows [t_begin, t_end) for token
  // 2v+1 and [t_begin, pad) for token 2v (pad >= t_begin), and its two partial
  // slots are slot and slot + 1, so each row's slots lie two apart (the reduce
  // entry's pad holds that stride). Sequences without KV rows keep one item
  // per token, marked pad = -1.
  int64_t Qu = 0;
  bool uniform = true;
  for (int b = 0; b < batch; ++b) {
    if (ngran[(size_t)b] == 0 || n_queries(b) == 0) continue;
    if (Qu == 0) Qu = n_queries(b);
    else if (n_queries(b) != Qu) uniform = false;
  }
  const bool pairs = opt.token_pairs && uniform && Qu >= 2 && Qu % 2 == 0;
  out->token_pairs = pairs;
  const int64_t Qn = pairs ? Qu / 2 : Qu;  // query units (tokens, or token pairs) of a sequence with rows
  const bool token_par = opt.token_parallel && uniform && Qn > 1 && max_ctas / Qn >= 1;
  if (token_par) max_ctas /= Qn;
  // query units per range
  auto weight = [&](int b) { return token_par ? (int64_t)1 : pairs ? n_queries(b) / 2 : n_queries(b); };
  int64_t U = 0, n_pieces_min = 0;
  for (int b = 0; b < batch; ++b) {
    U += ngran[(size_t)b] * weight(b);
    if (ngran[(size_t)b] > 0 && n_queries(b) > 0) n_pieces_min += weight(b);
  }
  // Greedy fill for a largest range cost T: the number of ranges it needs and,
  // when starts is given, the row where each range after the first begins. A
  // piece of a split sequence is min_granules long at least: a range that
  // could take less closes first, and a remainder shorter than that stays in
  // the range that holds the rest (which may then exceed T).
  auto fill = [&](int64_t T, std::vector<int64_t>* starts) {
    int64_t n = 1, cur = 0;
    bool empty = true;
    auto close = [&](int b, int64_t rem) {
      ++n;
      cur = 0;
      empty = true;
      if (starts) starts->push_back(tok[(size_t)b] + (ngran[(size_t)b] - rem) * G);
    };
    for (int b = 0; b < batch; ++b) {
      const int64_t w = weight(b) * kUnit, a = weight(b) * item_cost;
      int64_t rem = ngran[(size_t)b];
      if (rem == 0 || w == 0) continue;
      while (rem > 0) {
        int64_t fit = T > cur + a ? (T - cur - a) / w : 0;
        if (!empty && fit < std::min(rem, min_granules)) {
          close(b, rem);
          fit = T > a ? (T - a) / w : 0;
        }
        int64_t take = std::max<int64_t>(std::min(rem, fit), std::min(rem, min_granules));
        if (rem - take > 0 && rem - take < min_granules) take = rem;
        cur += a + take * w;
        empty = false;
        rem -= take;
        if (rem > 0) close(b, rem);
      }
    }
    return n;
  };
  std::vector<int64_t> cuts{0};
  if (U > 0) {
    // smallest T whose greedy fill needs at most max_ctas ranges, and ranges of min_granules at least
    int64_t lo = std::max<int64_t>((U * kUnit + max_ctas - 1) / max_ctas, 1);
    lo = std::max<int64_t>(lo, min_granules * kUnit);
    int64_t hi = std::max<int64_t>(U * kUnit + n_pieces_min * item_cost * 2 + item_cost, lo);
    while (fill(hi, nullptr) > max_ctas) hi *= 2;
    while (lo < hi) {
      const int64_t mid = lo + (hi - lo) / 2;
      if (fill(mid, nullptr) <= max_ctas) hi = mid; else lo = mid + 1;
    }
    fill(lo, &cuts);
  }
  cuts.push_back(total);
  const int64_t n_ranges = (int64_t)cuts.size() - 1;
  std::vector<std::pair<int64_t, int64_t>> ranges;  // non-empty CTA row ranges, in order
  for (int64_t k = 0; k < n_ranges; ++k)
    if (cuts[(size_t)k + 1] > cuts[(size_t)k]) ranges.emplace_back(cuts[(size_t)k], cuts[(size_t)k + 1]);
  if (ranges.empty()) ranges.emplace_back(0, 0);  // no rows at all: one CTA writes the zero outputs

  std::vector<WorkItem> items;
  std::vector<int32_t> cta_of_item;
  items.reserve((size_t)qo[(size_t)batch] + ranges.size() * 2);
  size_t cta = 0;  // range index
  const size_t last = ranges.size() - 1;
  // unit: the query token (or pair) index that picks the CTA of a token-parallel range
  auto push = [&](int b, int64_t t0, int64_t t1, int64_t j, int64_t unit, int64_t pad) {
    items.push_back(WorkItem{b, (int32_t)t0, (int32_t)t1, -1, (int32_t)seq_len(b), (int32_t)(qo[(size_t)b] + j),
                             (int32_t)j, (int32_t)pad});
    // token-parallel: the unit's CTA of the range. Only a sequence without KV rows can
    // have more than Qn units (its items write zeros); they go to the range's last CTA.
    cta_of_item.push_back((int32_t)(token_par ? (int64_t)cta * Qn + std::min<int64_t>(unit, Qn - 1) : (int64_t)cta));
  };
  for (int b = 0; b < batch; ++b) {
    const int64_t S = tok[(size_t)b], E = tok[(size_t)b + 1], q_b = n_queries(b);
    while (cta < last && ranges[cta].second <= S) ++cta;
    const bool pair_seq = pairs && S < E;  // a sequence with rows: its q_b is the even Qu
    // query tokens that see no KV token write zeros (a zero-row item; a pair when neither token sees one)
    if (pair_seq) {
      for (int64_t v = 0; v < q_b / 2; ++v)
        if (visible(b, 2 * v + 1) == 0) push(b, 0, 0, 2 * v, v, 0);
    } else {
      for (int64_t j = 0; j < q_b; ++j)
        if (visible(b, j) == 0) push(b, 0, 0, j, j, pairs ? -1 : 0);
    }
    if (S == E || q_b == 0) continue;
    while (true) {
      const int64_t a = std::max(S, ranges[cta].first) - S, e = std::min(E, ranges[cta].second) - S;
      if (pair_seq) {
        for (int64_t v = 0; v < q_b / 2; ++v) {  // token 2v+1 sees at least the rows token 2v sees
          const int64_t e1 = std::min(e, visible(b, 2 * v + 1));
          if (e1 > a) push(b, a, e1, 2 * v, v, std::max(a, std::min(e, visible(b, 2 * v))));
        }
      } else {
        for (int64_t j = 0; j < q_b; ++j) {  // the query tokens of this row range, back to back
          const int64_t ej = std::min(e, visible(b, j));
          if (ej > a) push(b, a, ej, j, j, 0);
        }
      }
      if (E <= ranges[cta].second || cta == last) break;
      ++cta;
    }
  }
  const int64_t used_ctas = (int64_t)ranges.size() * (token_par ? Qn : 1);
  if (token_par) {  // group the items by CTA, keeping each CTA's items (and each row's pieces) in order
    std::vector<size_t> order(items.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](size_t x, size_t y) { return cta_of_item[x] < cta_of_item[y]; });
    std::vector<WorkItem> sorted_items(items.size());
    std::vector<int32_t> sorted_cta(items.size());
    for (size_t i = 0; i < order.size(); ++i) {
      sorted_items[i] = items[order[i]];
      sorted_cta[i] = cta_of_item[order[i]];
    }
    items.swap(sorted_items);
    cta_of_item.swap(sorted_cta);
  }

  // Partial slots for query rows cut into several items, consecutive per row, rows in order.
  // A pair's two rows have the same items; their slots interleave (stride 2).
  const size_t n_rows = (size_t)qo[(size_t)batch];
  auto is_pair = [&](const WorkItem& w) { return pairs && w.pad >= 0; };
  std::vector<int32_t> count(n_rows, 0), next(n_rows, 0);
  std::vector<char> second(n_rows, 0);  // the second row of a pair
  for (const WorkItem& w : items) {
    count[(size_t)w.q_row]++;
    if (is_pair(w)) second[(size_t)w.q_row + 1] = 1;
  }
  std::vector<ReduceEntry> reduce;
  int slot = 0;
  for (size_t r = 0; r < n_rows; ++r) {
    if (count[r] <= 1 || second[r]) continue;
    next[r] = slot;
    if (r + 1 < n_rows && second[r + 1]) {
      reduce.push_back(ReduceEntry{(int32_t)r, slot, count[r], 2});
      reduce.push_back(ReduceEntry{(int32_t)r + 1, slot + 1, count[r], 2});
      slot += 2 * count[r];
    } else {
      reduce.push_back(ReduceEntry{(int32_t)r, slot, count[r], 0});
      slot += count[r];
    }
  }
  for (WorkItem& w : items)
    if (count[(size_t)w.q_row] > 1) {
      w.slot = next[(size_t)w.q_row];
      next[(size_t)w.q_row] += is_pair(w) ? 2 : 1;
    }

  // Items are already grouped by CTA in increasing order: CSR offsets.
  for (int32_t c : cta_of_item)
    if (c < 0 || (int64_t)c >= used_ctas) return MLA_ERR_ARG;  // not reached: every item has a CTA of the grid
  std::vector<int32_t> indptr((size_t)used_ctas + 1, 0);
  for (size_t i = 0; i < items.size(); ++i) indptr[(size_t)cta_of_item[i] + 1]++;
  for (int64_t c = 0; c < used_ctas; ++c) indptr[(size_t)c + 1] += indptr[(size_t)c];
  int64_t max_rows = 0;
  for (int64_t c = 0; c < used_ctas; ++c) {
    int64_t r = 0;
    for (int32_t i = indptr[(size_t)c]; i < indptr[(size_t)c + 1]; ++i) r += items[(size_t)i].t_end - items[(size_t)i].t_begin;
    max_rows = std::max(max_rows, r);
  }

  out->num_ctas = (int)used_ctas;
  out->num_slots = slot;
  out->n_items = (int)items.size();
  out->n_reduce = (int)reduce.size();
  out->max_rows_per_cta = max_rows;
  out->items = (WorkItem*)std::malloc(sizeof(WorkItem) * std::max<size_t>(items.size(), 1));
  out->work_indptr = (int32_t*)std::malloc(sizeof(int32_t) * indptr.size());
  out->reduce = (ReduceEntry*)std::malloc(sizeof(ReduceEntry) * std::max<size_t>(reduce.size(), 1));
  if (!out->items || !out->work_indptr || !out->reduce) {
    free_host_plan(out);
    return MLA_ERR_NOMEM;
  }
  if (!items.empty()) std::memcpy(out->items, items.data(), sizeof(WorkItem) * items.size());
  std::memcpy(out->work_indptr, indptr.data(), sizeof(int32_t) * indptr.size());
  if (!reduce.empty()) std::memcpy(out->reduce, reduce.data(), sizeof(ReduceEntry) * reduce.size());
  return MLA_OK;
}

// One query row per sequence.
std::vector<int64_t> single_queries(int batch) {
  std::vector<int64_t> qo((size_t)batch + 1);
  for (int b = 0; b <= batch; ++b) qo[(size_t)b] = b;
  return qo;
}

// Token offsets of the paged layout: (pages - 1) * page_size + last page length per sequence.
int paged_tokens(int batch, const int32_t* kv_indptr, const int32_t* last_page_len, int page_size,
                 std::vector<int64_t>* tok) {
  tok->assign((size_t)batch + 1, 0);
  for (int b = 0; b < batch; ++b) {
    const int64_t pages = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    int64_t n = 0;
    if (pages > 0) {
      const int64_t last = page_size > 1 ? (int64_t)last_page_len[b] : 1;
      if (last < 1 || last > page_size) return MLA_ERR_INDPTR;
      n = (pages - 1) * page_size + last;
      if (n > INT32_MAX) return MLA_ERR_INDPTR;  // token offsets inside a sequence are 32-bit
    }
    (*tok)[(size_t)b + 1] = (*tok)[(size_t)b] + n;
  }
  return MLA_OK;
}

int check_common(int batch, const int32_t* kv_indptr, int num_sms, const PlanOptions& opt, HostPlan* out) {
  if (batch < 0 || num_sms <= 0 || !out || (batch > 0 && !kv_indptr)) return MLA_ERR_ARG;
  if (opt.granularity <= 0 || opt.min_rows_per_split <= 0 || opt.ctas_per_sm <= 0) return MLA_ERR_ARG;
  *out = HostPlan{};
  out->batch = batch;
  if (batch > 0 && kv_indptr[0] != 0) return MLA_ERR_INDPTR;
  for (int b = 0; b < batch; ++b)
    if (kv_indptr[b + 1] < kv_indptr[b]) return MLA_ERR_INDPTR;
  return MLA_OK;
}

}  // namespace

int build_host_plan(int batch, const int32_t* kv_indptr, int num_sms, const PlanOptions& opt, HostPlan* out) {
  const int rc = check_common(batch, kv_indptr, num_sms, opt, out);
  if (rc != MLA_OK) return rc;
  std::vector<int64_t> tok((size_t)batch + 1, 0);
  for (int b = 1; b <= batch; ++b) tok[(size_t)b] = kv_indptr[b];
  return plan_tokens(batch, tok, single_queries(batch), false, num_sms, opt, out);
}

int build_host_plan_paged(int batch, const int32_t* kv_indptr, const int32_t* last_page_len, int page_size,
                          int num_sms, const PlanOptions& opt, HostPlan* out) {
  if (page_size < 1 || (batch > 0 && page_size > 1 && !last_page_len)) return MLA_ERR_ARG;
  int rc = check_common(batch, kv_indptr, num_sms, opt, out);
  if (rc != MLA_OK) return rc;
  std::vector<int64_t> tok;
  rc = paged_tokens(batch, kv_indptr, last_page_len, page_size, &tok);
  if (rc != MLA_OK) return rc;
  return plan_tokens(batch, tok, single_queries(batch), false, num_sms, opt, out);
}

int build_host_plan_multi(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* last_page_len, int page_size, bool causal, int num_sms,
                          const PlanOptions& opt, HostPlan* out) {
  if (page_size < 1 || (batch > 0 && (!qo_indptr || (page_size > 1 && !last_page_len)))) return MLA_ERR_ARG;
  int rc = check_common(batch, kv_indptr, num_sms, opt, out);
  if (rc != MLA_OK) return rc;
  if (batch > 0 && qo_indptr[0] != 0) return MLA_ERR_INDPTR;
  std::vector<int64_t> qo((size_t)batch + 1, 0);
  for (int b = 0; b < batch; ++b) {
    if (qo_indptr[b + 1] < qo_indptr[b]) return MLA_ERR_INDPTR;
    qo[(size_t)b + 1] = qo_indptr[b + 1];
  }
  std::vector<int64_t> tok;
  rc = paged_tokens(batch, kv_indptr, last_page_len, page_size, &tok);
  if (rc != MLA_OK) return rc;
  return plan_tokens(batch, tok, qo, causal, num_sms, opt, out);
}

}  // namespace mla
