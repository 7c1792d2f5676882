// Random inputs for the host split-KV planners (row, paged and multi-token
// layouts, extreme options, and the fixed-capacity planner of
// mla_decode_noalloc). Built with -fsanitize=address,undefined by
// tests/test_planner_fuzz.py; checks the work list, CSR and reduce map, and
// that the row-layout plans cover every row of every sequence exactly once.
#include <cstdio>
#include <cstdlib>
#include <memory>
#include <random>
#include <vector>
#include "internal.h"
#include "noalloc_plan.h"
using namespace mla;

// Row-layout plan check: the items of each sequence are consecutive, in CTA
// order, and cover [0, L_b) exactly once from the start; an empty sequence has
// one empty item; a sequence of several items owns one reduce entry whose
// consecutive slots the items take in order, a one-item sequence writes its
// output directly (slot -1). Returns an error message or nullptr.
static const char* check_rows(int B, const int32_t* ip, const WorkItem* items, int n_items, const int32_t* indptr,
                              int n_ctas, const ReduceEntry* red, int n_reduce, int n_slots) {
  if (n_ctas < 1 || indptr[0] != 0 || indptr[n_ctas] != n_items) return "csr ends";
  for (int c = 0; c < n_ctas; ++c)
    if (indptr[c + 1] < indptr[c]) return "csr order";
  std::vector<int> red_of(B, -1);
  for (int r = 0; r < n_reduce; ++r) {
    if (red[r].b < 0 || red[r].b >= B || red_of[red[r].b] >= 0) return "reduce entry";
    if (red[r].slot_begin < 0 || red[r].n_slots < 2 || red[r].slot_begin + red[r].n_slots > n_slots)
      return "reduce slots";
    red_of[red[r].b] = r;
  }
  int i = 0, prev_b = -1;
  while (i < n_items) {
    const int b = items[i].b;
    if (b <= prev_b || b >= B) return "sequence order";
    int j = i;
    int32_t t = 0;
    const int32_t L = ip[b + 1] - ip[b];
    while (j < n_items && items[j].b == b) {
      const WorkItem& w = items[j];
      if (w.t_begin != t || w.t_end < w.t_begin || w.seq_len != L || w.q_row != b || w.q_tok != 0) return "item";
      if (w.t_end == w.t_begin && L > 0) return "empty item";
      t = w.t_end;
      ++j;
    }
    if (t != L) return "coverage";
    if (j - i == 1) {
      if (items[i].slot != -1 || red_of[b] >= 0) return "whole sequence slot";
    } else {
      const int r = red_of[b];
      if (r < 0 || red[r].n_slots != j - i) return "split sequence reduce";
      for (int k = i; k < j; ++k)
        if (items[k].slot != red[r].slot_begin + (k - i)) return "slot order";
    }
    prev_b = b;
    i = j;
  }
  if (prev_b != B - 1 && B > 0) {
    // every sequence must appear
    return "missing sequence";
  }
  return nullptr;
}

int main(int argc, char** argv) {
  std::mt19937_64 rng(argc > 1 ? atoll(argv[1]) : 1);
  auto U = [&](int64_t lo, int64_t hi) { return (int64_t)(lo + rng() % (uint64_t)(hi - lo + 1)); };
  int ok = 0, err = 0;
  const int iters = argc > 2 ? atoi(argv[2]) : 20000;
  for (int iter = 0; iter < iters; ++iter) {
    const int B = (int)U(0, 40);
    PlanOptions o;
    o.granularity = (int)std::vector<int64_t>{1, 7, 16, 64, 128, 1000}[U(0, 5)];
    o.min_rows_per_split = (int)std::vector<int64_t>{1, 16, 128, 999, 100000}[U(0, 4)];
    o.ctas_per_sm = (int)U(1, 3);
    o.item_cost_rows = (int)std::vector<int64_t>{0, 1, 256, 100000}[U(0, 3)];
    o.token_parallel = U(0, 1) == 1;
    o.token_pairs = U(0, 1) == 1;
    const int num_sms = (int)U(1, 300);
    const int ps = (int)std::vector<int64_t>{1, 2, 3, 8, 64, 128, 1000}[U(0, 6)];
    std::vector<int32_t> ip(B + 1, 0), last(B, 1), qo(B + 1, 0);
    const int Qeq = (int)U(1, 6);
    for (int b = 0; b < B; ++b) {
      const int64_t pages = U(0, 1) ? U(0, 30) : 0;
      ip[b + 1] = ip[b] + (int32_t)pages;
      last[b] = (int32_t)U(1, ps);
      qo[b + 1] = qo[b] + (int32_t)(U(0, 3) == 0 ? U(0, 9) : Qeq);
    }
    HostPlan h;
    int rc;
    const int kind = (int)U(0, 2);
    if (kind == 0) rc = build_host_plan(B, ip.data(), num_sms, o, &h);
    else if (kind == 1) rc = build_host_plan_paged(B, ip.data(), last.data(), ps, num_sms, o, &h);
    else rc = build_host_plan_multi(B, qo.data(), ip.data(), last.data(), ps, U(0, 1) == 1, num_sms, o, &h);
    if (rc != 0) { ++err; continue; }
    ++ok;
    // structural checks: CSR within the items, slots within num_slots, reduce entries in range
    if (h.work_indptr[0] != 0 || h.work_indptr[h.num_ctas] != h.n_items) { printf("bad csr\n"); return 1; }
    for (int c = 0; c < h.num_ctas; ++c)
      if (h.work_indptr[c + 1] < h.work_indptr[c]) { printf("bad csr order\n"); return 1; }
    if (h.num_ctas > num_sms * o.ctas_per_sm && h.num_ctas > 1) { printf("too many ctas %d > %d\n", h.num_ctas, num_sms * o.ctas_per_sm); return 1; }
    for (int i = 0; i < h.n_items; ++i) {
      const WorkItem& w = h.items[i];
      if (w.slot >= h.num_slots || w.t_begin > w.t_end || w.t_begin < 0) { printf("bad item\n"); return 1; }
      // a token pair writes slots slot and slot + 1, and its first token's rows end within the item's
      if (h.token_pairs && w.pad >= 0) {
        if (w.slot >= 0 && w.slot + 1 >= h.num_slots) { printf("bad pair slot\n"); return 1; }
        if (w.t_end > w.t_begin && (w.pad < w.t_begin || w.pad > w.t_end)) { printf("bad pair end\n"); return 1; }
      }
    }
    for (int r = 0; r < h.n_reduce; ++r) {  // slots slot_begin + k * stride, k < n_slots
      const int stride = h.reduce[r].pad > 1 ? h.reduce[r].pad : 1;
      if (h.reduce[r].slot_begin < 0 || h.reduce[r].slot_begin + stride * (h.reduce[r].n_slots - 1) >= h.num_slots) {
        printf("bad reduce\n");
        return 1;
      }
    }
    if (kind == 0) {
      const char* e = check_rows(B, ip.data(), h.items, h.n_items, h.work_indptr, h.num_ctas, h.reduce, h.n_reduce,
                                 h.num_slots);
      if (e) { printf("row plan: %s (iter %d)\n", e, iter); return 1; }
    }
    free_host_plan(&h);
  }

  // The fixed-capacity planner of mla_decode_noalloc: up to its batch limit,
  // lengths from empty to long, any SM count.
  auto fp = std::make_unique<noalloc::FixedPlan>();
  int fixed_ok = 0, fixed_limit = 0;
  for (int iter = 0; iter < iters / 4; ++iter) {
    const int B = (int)(U(0, 3) == 0 ? U(0, noalloc::kMaxBatch) : U(0, 70));
    const int num_sms = (int)std::vector<int64_t>{1, 2, 7, 148, 152, 1024, 5000}[U(0, 6)];
    const int64_t max_len = std::vector<int64_t>{1, 200, 9000, 300000}[U(0, 3)];
    std::vector<int32_t> ip(B + 1, 0);
    for (int b = 0; b < B; ++b) ip[b + 1] = ip[b] + (int32_t)(U(0, 4) == 0 ? 0 : U(0, max_len));
    const int rc = noalloc::plan_fixed(B, ip.data(), num_sms, fp.get());
    if (rc == MLA_ERR_NOALLOC_LIMIT) { ++fixed_limit; continue; }
    if (rc != MLA_OK) { printf("fixed plan: rc %d\n", rc); return 1; }
    ++fixed_ok;
    if (B == 0) continue;
    if (fp->n_ctas > std::min(num_sms, noalloc::kMaxCtas)) { printf("fixed plan: %d ctas\n", fp->n_ctas); return 1; }
    if (fp->n_items > noalloc::kMaxItems || fp->n_slots > noalloc::kMaxSlots || fp->n_reduce > noalloc::kMaxReduce) {
      printf("fixed plan: capacity\n");
      return 1;
    }
    const char* e = check_rows(B, ip.data(), fp->items, fp->n_items, fp->indptr, fp->n_ctas, fp->reduce,
                               fp->n_reduce, fp->n_slots);
    if (e) { printf("fixed plan: %s (iter %d, B %d, sms %d)\n", e, iter, B, num_sms); return 1; }
    // balance: no CTA holds more than the even share of 64-row granules, rounded up,
    // and at least one granule when there are rows
    int64_t granules = 0;
    for (int b = 0; b < B; ++b) granules += (ip[b + 1] - ip[b] + 63) / 64;
    const int64_t share = std::max<int64_t>(1, (granules + std::min(num_sms, noalloc::kMaxCtas) - 1) /
                                                   std::min(num_sms, noalloc::kMaxCtas));
    for (int c = 0; c < fp->n_ctas; ++c) {
      int64_t g = 0;
      for (int i = fp->indptr[c]; i < fp->indptr[c + 1]; ++i)
        g += (fp->items[i].t_end - fp->items[i].t_begin + 63) / 64;
      if (g > share + 1) { printf("fixed plan: cta %d holds %lld granules, share %lld\n", c, (long long)g, (long long)share); return 1; }
    }
  }
  printf("ok %d err %d fixed %d limit %d\n", ok, err, fixed_ok, fixed_limit);
  return 0;
}
