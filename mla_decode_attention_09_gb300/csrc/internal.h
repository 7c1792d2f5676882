// Internal declarations shared by the planner, the C ABI and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

#include "mla_decode.h"

namespace mla {

constexpr int kHeads = MLA_NUM_HEADS;     // 16 query heads share one KV head
constexpr int kQkDim = MLA_QK_HEAD_DIM;   // 576 = 512 latent + 64 rope
constexpr int kVDim = MLA_V_HEAD_DIM;     // 512: value = first 512 entries of the KV row

// One unit of stage-1 work: rows [t_begin, t_end) of sequence b (row offsets
// relative to the sequence start). slot >= 0: write normalised fp32 partial O
// and LSE to workspace slot `slot`; slot < 0: the item covers the whole
// sequence and writes final bf16 output. seq_len is the length the plan saw,
// checked against the device kv_indptr.
struct WorkItem {
  int32_t b;
  int32_t t_begin;
  int32_t t_end;
  int32_t slot;
  int32_t seq_len;
  int32_t pad[3];
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// One split sequence for the reduce: slots [slot_begin, slot_begin + n_slots).
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
  WorkItem* items = nullptr;     // [n_items]
  int n_items = 0;
  int32_t* work_indptr = nullptr;  // [num_ctas + 1]
  ReduceEntry* reduce = nullptr;   // [n_reduce]
  int n_reduce = 0;
};

// Resolved planner options (defaults applied).
struct PlanOptions {
  int64_t num_kv_slots = 0;
  int min_rows_per_split = 256;
  int granularity = 128;  // the tcgen05 kernel's tile height (a multiple of the warp-level kernels' 64)
  int ctas_per_sm = 1;
  int fp8_kernel = 0;  // 0 = tcgen05 / TMA kernel, 1 = warp-level mma.sync kernel
};

PlanOptions resolve_options(const mla_plan_options* o);

// Pure host planning (no CUDA calls). Returns MLA_OK or an error; on success
// the arrays in *out are malloc'ed and must be freed with free_host_plan.
int build_host_plan(int batch, const int32_t* kv_indptr, int num_sms, const PlanOptions& opt, HostPlan* out);
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
  int fp8_kernel;        // see PlanOptions
};

struct DecodeArgs {
  const void* q;
  const void* kv;
  const float* kv_scale;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  void* out;
  float sm_scale;
};

// Kernel launchers (stage1.cu / reduce.cu). Return cudaError_t as int.
int launch_stage1(int dtype_mode, const DecodeArgs& a, const DevicePlan& p, const void* zero_row, void* stream);
int launch_reduce(void* out, const DevicePlan& p, void* stream, bool pdl);
int launch_stage1_fp8_umma(const DecodeArgs& a, const DevicePlan& p, void* stream);

}  // namespace mla
