// Random inputs for the host split-KV planners (row, paged and multi-token
// layouts, extreme options). Built with -fsanitize=address,undefined by
// tests/test_planner_fuzz.py; checks the work list, CSR and reduce map.
#include <cstdio>
#include <cstdlib>
#include <random>
#include <vector>
#include "internal.h"
using namespace mla;
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
    }
    for (int r = 0; r < h.n_reduce; ++r)
      if (h.reduce[r].slot_begin < 0 || h.reduce[r].slot_begin + h.reduce[r].n_slots > h.num_slots) { printf("bad reduce\n"); return 1; }
    free_host_plan(&h);
  }
  printf("ok %d err %d\n", ok, err);
  return 0;
}
