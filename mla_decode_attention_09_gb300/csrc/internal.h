// Internal declarations shared by the planner, the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "mla_decode.h"

namespace mla {

constexpr int kHeads = MLA_NUM_HEADS;     // 16 query heads share one KV head
constexpr int kQkDim = MLA_QK_HEAD_DIM;   // 576 = 512 latent + 64 rope
constexpr int kVDim = MLA_V_HEAD_DIM;     // 512: value = first 512 entries of the KV row

// One unit of stage-1 work: query row q_row attends to KV tokens
// [t_begin, t_end) of sequence b (offsets relative to the sequence start).
// slot >= 0: write normalised fp32 partial O and LSE to workspace slot
// `slot`; slot < 0: the item covers every token the query row sees and writes
// its final bf16 output. seq_len is the token count the plan saw, checked
// against the device kv_indptr (and last page lengths); q_tok is the query
// token's index within its sequence, checked against the device qo_indptr.
// Single-token plans have q_row = b and q_tok = 0. pad is 0, except in
// token-pair plans: there an item with pad >= 0 covers query rows q_row and
// q_row + 1 (tokens q_tok, q_tok + 1), the first over [t_begin, pad), the
// second over [t_begin, t_end), with partial slots slot and slot + 1; pad = -1
// marks a single-token item (a sequence without KV rows).
struct WorkItem {
  int32_t b;
  int32_t t_begin;
  int32_t t_end;
  int32_t slot;
  int32_t seq_len;
  int32_t q_row;
  int32_t q_tok;
  int32_t pad;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// One split query row for the reduce: n_slots slots from slot_begin, pad apart
// (0 or 1: consecutive; 2: a row of a token pair), merged into output row b.
struct ReduceEntry {
  int32_t b;
  int32_t slot_begin;
  int32_t n_slots;
  int32_t pad;
};
static_assert(sizeof(ReduceEntry) == 16, "ReduceEntry layout");

// Host planning result.
struct HostPlan {
  int batch = 0;
  int num_ctas = 0;
  int num_slots = 0;
  int64_t total_rows = 0;
  int64_t max_rows_per_cta = 0;
  bool token_pairs = false;  // items are token pairs (see plan_tokens)
  WorkItem* items = nullptr;     // [n_items]
  int n_items = 0;
  int32_t* work_indptr = nullptr;  // [num_ctas + 1]
  ReduceEntry* reduce = nullptr;   // [n_reduce]
  int n_reduce = 0;
};

// Resolved planner options (defaults applied).
struct PlanOptions {
  int64_t num_kv_slots = 0;
  // 64 rows: the warp-level kernels' tile, half a tcgen05 tile. Measured against 128 (graph-timed,
  // inputs rotated out of L2): bf16 B=4 kv_len=1024 12.6 -> 11.2 us (64 CTAs instead of 32), bf16
  // ragged B=128 117.6 -> 116.8 us, the fp8 workloads unchanged within 0.1-0.5 us.
  int min_rows_per_split = 64;
  int granularity = 64;
  int ctas_per_sm = 1;
  int fp8_kernel = 0;  // 0 = tcgen05 / TMA kernel, 1 = warp-level mma.sync kernel
  int fp8_issuers = 0;  // tcgen05 kernel: 0 or 2 two MMA-issuing threads, 1 one issuer + three loaders
  int item_cost_rows = 256;  // balancing cost of each item a CTA starts, in KV rows (0 = none)
  bool token_parallel = true;  // multi-token plans with equal query counts: one CTA per (range, token)
  bool token_pairs = false;    // multi-token plans with equal even query counts: tokens in pairs, one pass each
};

// Two MMA-issuing threads in the tcgen05 kernel unless asked for one: one
// issuer frees a warp for a third row loader, which pays only when every
// tile is copied row by row from rows scattered one by one.
inline bool dual_issue(const PlanOptions& o) { return o.fp8_issuers != 1; }

PlanOptions resolve_options(const mla_plan_options* o);

// Pure host planning (no CUDA calls). Returns MLA_OK or an error; on success
// the arrays in *out are malloc'ed and must be freed with free_host_plan.
// Row addressing: sequence b holds kv_indptr[b+1] - kv_indptr[b] tokens.
int build_host_plan(int batch, const int32_t* kv_indptr, int num_sms, const PlanOptions& opt, HostPlan* out);
// Paged addressing: kv_indptr counts pages of page_size tokens and
// last_page_len[b] (1..page_size) gives the tokens used in b's last page.
int build_host_plan_paged(int batch, const int32_t* kv_indptr, const int32_t* last_page_len, int page_size,
                          int num_sms, const PlanOptions& opt, HostPlan* out);
// Several query tokens per sequence: rows qo_indptr[b] .. qo_indptr[b+1]-1 of
// q and out. With causal, query token j of a sequence with q_b query tokens
// and L_b KV tokens sees its first max(0, L_b - q_b + j + 1) tokens; else all.
// KV addressing as build_host_plan_paged (page_size 1 = row addressing,
// last_page_len may then be NULL).
int build_host_plan_multi(int batch, const int32_t* qo_indptr, const int32_t* kv_indptr,
                          const int32_t* last_page_len, int page_size, bool causal, int num_sms,
                          const PlanOptions& opt, HostPlan* out);
void free_host_plan(HostPlan* p);

// Device-side view of a plan, passed to the kernels by value.
struct DevicePlan {
  const WorkItem* items;
  const int32_t* work_indptr;
  const ReduceEntry* reduce;
  float* part_o;     // [num_slots, 16, 512] fp32, normalised partial output
  float* part_lse;   // [num_slots, 16] fp32, log2-domain LSE of the partial
  int* err;          // first error status recorded by a kernel (0 = none)
  int64_t num_kv_slots;  // 0 = unchecked
  int num_ctas;
  int n_reduce;
  int reduce_max_slots;  // most partial slots of any reduce entry (picks the reduce instance)
  int fp8_kernel;        // see PlanOptions
  int dual_issue;        // tcgen05 kernel instance: 1 two MMA issuers, 0 one
  int token_pairs;       // the items are token pairs (only the fp8 tensor-core pair kernel takes them)
};

struct DecodeArgs {
  const void* q;
  const void* kv;
  const float* kv_scale;
  const int32_t* kv_indptr;   // per sequence: offsets into kv_indices (pages when page_size > 1)
  const int32_t* kv_indices;  // KV row of each token, or page id of each page when page_size > 1
  void* out;
  float sm_scale;
  const int32_t* kv_last_page_len = nullptr;  // [B], tokens used in each last page (page_size > 1)
  int page_size = 1;                          // tokens per page; 1 = every kv_indices entry is a row
  const int32_t* qo_indptr = nullptr;         // [B+1] query rows per sequence (multi-token plans)
  uint32_t page_magic = 1;                    // t / page_size = (mulhi(t, page_magic) + t) >> page_shift
  int page_shift = 0;
};

// Sets page_size and the constants that divide a token index by it with one
// multiply-high, an add and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(m, n) + n) >> l for
// 0 <= n < 2^32; for n < 2^31 the sum fits in 32 bits. The kernels' loaders
// divide every token of every tile, and a general integer division there (even
// a branch to one) measured ~20% slower.
inline void set_page_size(DecodeArgs& a, int page_size) {
  uint32_t l = 0;
  while ((1ull << l) < (uint64_t)page_size) ++l;
  a.page_size = page_size;
  a.page_shift = (int)l;
  a.page_magic = (uint32_t)(((1ull << 32) * ((1ull << l) - (uint64_t)page_size)) / (uint64_t)page_size + 1);
}

#ifdef __CUDACC__
// Token addressing, specialised at compile time: kPaged = false is the row
// layout (every kv_indices entry is a row, lengths are kv_indptr differences);
// kPaged = true takes pages of a.page_size tokens.
//
// Tokens of sequence b according to the device arrays: pages of page_size
// tokens, the last one holding kv_last_page_len[b]. -1 when that length lies
// outside [1, page_size] (the caller treats it like a plan mismatch).
template <bool kPaged>
__device__ __forceinline__ int64_t device_seq_tokens(const DecodeArgs& a, int b) {
  const int64_t pages = (int64_t)a.kv_indptr[b + 1] - a.kv_indptr[b];
  if (!kPaged || pages <= 0) return pages;
  const int last = a.kv_last_page_len[b];
  if (last < 1 || last > a.page_size) return -1;
  return (pages - 1) * a.page_size + last;
}
// The item's query row agrees with the device qo_indptr (always, for
// single-token calls, which pass none).
__device__ __forceinline__ bool item_query_ok(const DecodeArgs& a, const WorkItem& w) {
  return a.qo_indptr == nullptr || (int64_t)a.qo_indptr[w.b] + w.q_tok == w.q_row;
}
// kv_indices position (relative to the sequence's first entry) of token t.
template <bool kPaged>
__device__ __forceinline__ int token_entry(const DecodeArgs& a, int t) {
  if (!kPaged) return t;
  return (int)((__umulhi((uint32_t)t, a.page_magic) + (uint32_t)t) >> a.page_shift);
}
// KV row of token t given the kv_indices entry e that token_entry pointed at
// (entry * page_size + t % page_size), in 64 bits: a caller range-checks it.
template <bool kPaged>
__device__ __forceinline__ int64_t token_row(const DecodeArgs& a, int32_t e, int t) {
  if (!kPaged) return (int64_t)e;
  return (int64_t)e * a.page_size + (t - token_entry<true>(a, t) * a.page_size);
}
#endif

// Kernel launchers (stage1.cu / reduce.cu). Return cudaError_t as int.
int launch_stage1(int dtype_mode, const DecodeArgs& a, const DevicePlan& p, const void* zero_row, void* stream);
int launch_reduce(void* out, const DevicePlan& p, void* stream, bool pdl);
int launch_stage1_fp8_umma(const DecodeArgs& a, const DevicePlan& p, void* stream);
// a16w8 on the tensor cores: the bf16 query as two e4m3 terms (stage1_umma_a16.cu).
int launch_stage1_a16w8_umma(const DecodeArgs& a, const DevicePlan& p, void* stream);
// fp8 stage 1 of a token-pair plan: both tokens of each item in one pass over its rows
int launch_stage1_fp8_pairs_umma(const DecodeArgs& a, const DevicePlan& p, void* stream);

}  // namespace mla
