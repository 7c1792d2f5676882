// C ABI of the MLA decode library: plan lifetime and caching, argument
// validation, and the stage-1 / reduce launches. No exception leaves this file.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "internal.h"

struct mla_plan {
  int device = -1;
  int refcount = 0;
  int batch = 0;
  int num_sms = 0;
  mla::PlanOptions opt;
  int kind = 0;                  // Layout kind the plan was built for; serves only that decode call
  int page_size = 1;
  bool causal = false;
  std::vector<int32_t> indptr;   // cache key contents
  std::vector<int32_t> last_page_len;
  std::vector<int32_t> qo_indptr;
  mla::HostPlan host;
  mla::DevicePlan dev{};
  // Several query tokens: a second work list in token pairs, built unless the option turns it
  // off and only when the query counts allow it; fp8 decodes on the tensor-core kernel use it,
  // every other decode the first list. Both share the partial buffers and the error word.
  bool want_pairs = false;
  bool has_pairs = false;
  mla::HostPlan host_pairs;
  mla::DevicePlan dev_pairs{};
  void* block = nullptr;         // single device allocation backing every buffer
  size_t block_bytes = 0;
  const void* zero_row = nullptr;  // 1152 zero bytes (source for tail rows of a tile)
};

namespace {

std::mutex g_mu;
std::vector<mla_plan*> g_cache;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Layout a plan is built for, and that a decode call passes: row addressing
// (kRowsKind), pages of page_size tokens with last page lengths `last` (NULL
// when page_size is 1), or several query tokens per sequence (rows qo[b] ..
// qo[b+1]-1, causal or not) over either KV addressing. For plans the arrays
// are host copies; for decode calls, the device arrays.
enum { kRowsKind = 0, kPagedKind = 1, kMultiKind = 2 };
struct Layout {
  int kind;
  int page_size;
  const int32_t* last;
  const int32_t* qo;
  bool causal;
};

bool same_array(const std::vector<int32_t>& v, const int32_t* a, size_t n) {
  if (a == nullptr || n == 0) return v.empty();
  return v.size() == n && std::memcmp(v.data(), a, sizeof(int32_t) * n) == 0;
}

bool same_key(const mla_plan* p, int device, int batch, const int32_t* indptr, const Layout& l, int num_sms,
              const mla::PlanOptions& o, bool want_pairs) {
  return p->device == device && p->batch == batch && p->num_sms == num_sms && p->kind == l.kind &&
         p->page_size == l.page_size && p->causal == l.causal && p->opt.num_kv_slots == o.num_kv_slots &&
         p->opt.min_rows_per_split == o.min_rows_per_split && p->opt.granularity == o.granularity &&
         p->opt.ctas_per_sm == o.ctas_per_sm && p->opt.fp8_kernel == o.fp8_kernel &&
         p->opt.fp8_issuers == o.fp8_issuers && p->opt.item_cost_rows == o.item_cost_rows &&
         p->opt.token_parallel == o.token_parallel && p->want_pairs == want_pairs &&
         std::memcmp(p->indptr.data(), indptr, sizeof(int32_t) * (size_t)(batch + 1)) == 0 &&
         same_array(p->last_page_len, l.last, (size_t)batch) &&
         same_array(p->qo_indptr, l.qo, batch > 0 ? (size_t)batch + 1 : 0);
}

void destroy_plan(mla_plan* p) {
  if (p->block) {
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    cudaFree(p->block);
    if (cur != p->device && cur >= 0) cudaSetDevice(cur);
  }
  mla::free_host_plan(&p->host);
  mla::free_host_plan(&p->host_pairs);
  delete p;
}

int check_device(int* device_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MLA_ERR_DEVICE;
  if (major != 10 || minor != 3) return MLA_ERR_DEVICE;  // kernels are built for sm_103a only
  *device_out = dev;
  return MLA_OK;
}

int make_plan(int batch, const int32_t* kv_indptr_host, const Layout& l, int num_sms, const mla::PlanOptions& opt,
              bool want_pairs, int device, mla_plan** out) {
  mla_plan* p = new (std::nothrow) mla_plan();
  if (!p) return MLA_ERR_NOMEM;
  p->device = device;
  p->batch = batch;
  p->num_sms = num_sms;
  p->opt = opt;
  p->kind = l.kind;
  p->page_size = l.page_size;
  p->causal = l.causal;
  p->indptr.assign(kv_indptr_host, kv_indptr_host + batch + 1);
  if (l.last && batch > 0) p->last_page_len.assign(l.last, l.last + batch);
  if (l.qo && batch > 0) p->qo_indptr.assign(l.qo, l.qo + batch + 1);
  p->want_pairs = want_pairs;
  mla::PlanOptions opt_main = opt;
  opt_main.token_pairs = false;
  int rc = l.kind == kMultiKind
               ? mla::build_host_plan_multi(batch, l.qo, kv_indptr_host, l.last, l.page_size, l.causal, num_sms,
                                            opt_main, &p->host)
           : l.kind == kPagedKind ? mla::build_host_plan_paged(batch, kv_indptr_host, l.last, l.page_size, num_sms,
                                                               opt_main, &p->host)
                                  : mla::build_host_plan(batch, kv_indptr_host, num_sms, opt_main, &p->host);
  if (rc == MLA_OK && l.kind == kMultiKind && want_pairs) {
    mla::PlanOptions opt_pairs = opt;
    opt_pairs.token_pairs = true;
    rc = mla::build_host_plan_multi(batch, l.qo, kv_indptr_host, l.last, l.page_size, l.causal, num_sms, opt_pairs,
                                    &p->host_pairs);
    p->has_pairs = rc == MLA_OK && p->host_pairs.token_pairs;
    if (rc == MLA_OK && !p->has_pairs) mla::free_host_plan(&p->host_pairs);  // the counts do not pair up
  }
  if (rc != MLA_OK) {
    destroy_plan(p);
    return rc;
  }
  const mla::HostPlan& h = p->host;
  const mla::HostPlan& hp = p->host_pairs;
  const int slots = p->has_pairs ? std::max(h.num_slots, hp.num_slots) : h.num_slots;
  // layout of the single device block
  size_t off = 0;
  const size_t o_items = off;
  off = align_up(off + sizeof(mla::WorkItem) * (size_t)h.n_items, 256);
  const size_t o_indptr = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(h.num_ctas + 1), 256);
  const size_t o_reduce = off;
  off = align_up(off + sizeof(mla::ReduceEntry) * (size_t)h.n_reduce, 256);
  const size_t o_items_p = off;
  if (p->has_pairs) off = align_up(off + sizeof(mla::WorkItem) * (size_t)hp.n_items, 256);
  const size_t o_indptr_p = off;
  if (p->has_pairs) off = align_up(off + sizeof(int32_t) * (size_t)(hp.num_ctas + 1), 256);
  const size_t o_reduce_p = off;
  if (p->has_pairs) off = align_up(off + sizeof(mla::ReduceEntry) * (size_t)hp.n_reduce, 256);
  const size_t o_po = off;
  off = align_up(off + sizeof(float) * (size_t)slots * mla::kHeads * mla::kVDim, 256);
  const size_t o_lse = off;
  off = align_up(off + sizeof(float) * (size_t)slots * mla::kHeads, 256);
  const size_t o_err = off;
  off = align_up(off + sizeof(int), 256);
  const size_t o_zero = off;
  off = align_up(off + mla::kQkDim * 2, 256);
  p->block_bytes = off;
  if (cudaMalloc(&p->block, off) != cudaSuccess) {
    cudaGetLastError();
    p->block = nullptr;
    destroy_plan(p);
    return MLA_ERR_NOMEM;
  }
  char* base = static_cast<char*>(p->block);
  std::vector<char> staging(o_po, 0);  // work lists and reduce maps, uploaded in one copy
  if (h.n_items) std::memcpy(staging.data() + o_items, h.items, sizeof(mla::WorkItem) * (size_t)h.n_items);
  std::memcpy(staging.data() + o_indptr, h.work_indptr, sizeof(int32_t) * (size_t)(h.num_ctas + 1));
  if (h.n_reduce) std::memcpy(staging.data() + o_reduce, h.reduce, sizeof(mla::ReduceEntry) * (size_t)h.n_reduce);
  if (p->has_pairs) {
    if (hp.n_items) std::memcpy(staging.data() + o_items_p, hp.items, sizeof(mla::WorkItem) * (size_t)hp.n_items);
    std::memcpy(staging.data() + o_indptr_p, hp.work_indptr, sizeof(int32_t) * (size_t)(hp.num_ctas + 1));
    if (hp.n_reduce)
      std::memcpy(staging.data() + o_reduce_p, hp.reduce, sizeof(mla::ReduceEntry) * (size_t)hp.n_reduce);
  }
  if (cudaMemcpy(base, staging.data(), o_po, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(base + o_err, 0, off - o_err) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    destroy_plan(p);
    return MLA_ERR_CUDA;
  }
  p->dev.items = reinterpret_cast<const mla::WorkItem*>(base + o_items);
  p->dev.work_indptr = reinterpret_cast<const int32_t*>(base + o_indptr);
  p->dev.reduce = reinterpret_cast<const mla::ReduceEntry*>(base + o_reduce);
  p->dev.part_o = reinterpret_cast<float*>(base + o_po);
  p->dev.part_lse = reinterpret_cast<float*>(base + o_lse);
  p->dev.err = reinterpret_cast<int*>(base + o_err);
  p->dev.num_kv_slots = opt.num_kv_slots;
  p->dev.num_ctas = h.num_ctas;
  p->dev.n_reduce = h.n_reduce;
  p->dev.reduce_max_slots = 0;
  for (int i = 0; i < h.n_reduce; ++i) p->dev.reduce_max_slots = std::max(p->dev.reduce_max_slots, h.reduce[i].n_slots);
  p->dev.fp8_kernel = opt.fp8_kernel;
  p->dev.dual_issue = mla::dual_issue(opt) ? 1 : 0;
  p->dev.token_pairs = 0;
  if (p->has_pairs) {
    p->dev_pairs = p->dev;
    p->dev_pairs.items = reinterpret_cast<const mla::WorkItem*>(base + o_items_p);
    p->dev_pairs.work_indptr = reinterpret_cast<const int32_t*>(base + o_indptr_p);
    p->dev_pairs.reduce = reinterpret_cast<const mla::ReduceEntry*>(base + o_reduce_p);
    p->dev_pairs.num_ctas = hp.num_ctas;
    p->dev_pairs.n_reduce = hp.n_reduce;
    p->dev_pairs.reduce_max_slots = 0;
    for (int i = 0; i < hp.n_reduce; ++i)
      p->dev_pairs.reduce_max_slots = std::max(p->dev_pairs.reduce_max_slots, hp.reduce[i].n_slots);
    p->dev_pairs.token_pairs = 1;
  }
  p->zero_row = base + o_zero;
  p->refcount = 1;
  *out = p;
  return MLA_OK;
}

int validate_decode(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
                    const int32_t* kv_indices, const void* out, int dtype_mode, const mla_plan* plan,
                    const Layout& l) {
  if (!plan || plan->refcount <= 0) return MLA_ERR_ARG;
  if (plan->kind != l.kind || plan->page_size != l.page_size) return MLA_ERR_ARG;
  if (l.page_size > 1 && plan->batch > 0 && !l.last) return MLA_ERR_ARG;
  if (l.kind == kMultiKind && plan->batch > 0 && !l.qo) return MLA_ERR_ARG;
  if (dtype_mode != MLA_MODE_BF16 && dtype_mode != MLA_MODE_FP8 && dtype_mode != MLA_MODE_A16W8)
    return MLA_ERR_DTYPE;
  if (plan->batch > 0) {
    if (!q || !kv || !kv_indptr || !out) return MLA_ERR_ARG;
    if (plan->host.total_rows > 0 && !kv_indices) return MLA_ERR_ARG;
    if (dtype_mode != MLA_MODE_BF16 && !kv_scale) return MLA_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(out)) & 15)
      return MLA_ERR_ALIGN;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != plan->device) return MLA_ERR_DEVICE;
  return MLA_OK;
}

int plan_common(int batch, const int32_t* kv_indptr_host, const Layout& layout, int num_sms,
                const mla_plan_options* options, mla_plan** plan_out) {
  try {
    if (!plan_out || batch < 0 || (!kv_indptr_host && batch > 0)) return MLA_ERR_ARG;
    if (layout.page_size < 1 || (layout.page_size > 1 && batch > 0 && !layout.last)) return MLA_ERR_ARG;
    if (layout.kind == kMultiKind && batch > 0 && !layout.qo) return MLA_ERR_ARG;
    *plan_out = nullptr;
    int device = -1;
    int rc = check_device(&device);
    if (rc != MLA_OK) return rc;
    if (num_sms <= 0) {
      if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return MLA_ERR_CUDA;
    }
    const mla::PlanOptions opt = mla::resolve_options(options);
    // the token-pair list of a multi-token plan: on unless the option is negative
    const bool want_pairs = layout.kind == kMultiKind && !(options && options->token_pairs < 0);
    static const int32_t kZero = 0;
    const int32_t* indptr = batch > 0 ? kv_indptr_host : &kZero;
    std::lock_guard<std::mutex> lock(g_mu);
    for (mla_plan* p : g_cache) {
      if (same_key(p, device, batch, indptr, layout, num_sms, opt, want_pairs)) {
        ++p->refcount;
        *plan_out = p;
        return MLA_OK;
      }
    }
    mla_plan* p = nullptr;
    rc = make_plan(batch, indptr, layout, num_sms, opt, want_pairs, device, &p);
    if (rc != MLA_OK) return rc;
    g_cache.push_back(p);
    *plan_out = p;
    return MLA_OK;
  } catch (...) {
    return MLA_ERR_NOMEM;
  }
}

int decode_common(const mla::DecodeArgs& a, int dtype_mode, mla_plan* workspace, void* stream, bool reduce) {
  if (workspace->batch == 0) return MLA_OK;
  // fp8 on the tensor-core kernel takes the token-pair list when the plan has one
  const bool pairs = workspace->has_pairs && dtype_mode == MLA_MODE_FP8 && workspace->dev.fp8_kernel == 0;
  const mla::DevicePlan& dv = pairs ? workspace->dev_pairs : workspace->dev;
  const int rc = pairs ? mla::launch_stage1_fp8_pairs_umma(a, dv, stream)
                       : mla::launch_stage1(dtype_mode, a, dv, workspace->zero_row, stream);
  if (rc != 0) return MLA_ERR_CUDA;
  // the reduce is launched programmatically dependent: it starts while stage 1
  // drains and waits for its results on the device
  if (reduce && mla::launch_reduce(a.out, dv, stream, true) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}

constexpr Layout kRows{kRowsKind, 1, nullptr, nullptr, false};

}  // namespace

extern "C" {

int mla_decode_plan_ex(int batch, const int32_t* kv_indptr_host, int num_sms, const mla_plan_options* options,
                       mla_plan** plan_out) {
  return plan_common(batch, kv_indptr_host, kRows, num_sms, options, plan_out);
}

int mla_decode_plan_paged(int batch, const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                          int page_size, int num_sms, const mla_plan_options* options, mla_plan** plan_out) {
  const Layout l{kPagedKind, page_size, page_size > 1 ? kv_last_page_len_host : nullptr, nullptr, false};
  return plan_common(batch, kv_indptr_host, l, num_sms, options, plan_out);
}

int mla_decode_plan_multi(int batch, const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                          const int32_t* kv_last_page_len_host, int page_size, int causal, int num_sms,
                          const mla_plan_options* options, mla_plan** plan_out) {
  const Layout l{kMultiKind, page_size, page_size > 1 ? kv_last_page_len_host : nullptr, qo_indptr_host,
                 causal != 0};
  return plan_common(batch, kv_indptr_host, l, num_sms, options, plan_out);
}

int mla_decode_plan(int batch, const int32_t* kv_indptr_host, int num_sms, mla_plan** plan_out) {
  return mla_decode_plan_ex(batch, kv_indptr_host, num_sms, nullptr, plan_out);
}

int mla_plan_release(mla_plan* plan) {
  if (!plan) return MLA_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  for (size_t i = 0; i < g_cache.size(); ++i) {
    if (g_cache[i] == plan) {
      if (--plan->refcount == 0) {
        g_cache.erase(g_cache.begin() + (long)i);
        destroy_plan(plan);
      }
      return MLA_OK;
    }
  }
  return MLA_ERR_ARG;
}

int mla_plan_destroy(mla_plan* plan) { return mla_plan_release(plan); }

size_t mla_plan_workspace_bytes(const mla_plan* plan) { return plan ? plan->block_bytes : 0; }

int mla_plan_get_info(const mla_plan* plan, mla_plan_info* info) {
  if (!plan || !info) return MLA_ERR_ARG;
  info->batch = plan->batch;
  info->num_ctas = plan->host.num_ctas;
  info->num_work_items = plan->host.n_items;
  info->num_partial_slots = plan->host.num_slots;
  info->num_split_seqs = plan->host.n_reduce;
  info->device = plan->device;
  info->total_rows = plan->host.total_rows;
  info->max_rows_per_cta = plan->host.max_rows_per_cta;
  info->workspace_bytes = plan->block_bytes;
  info->token_pairs = plan->has_pairs ? 1 : 0;
  return MLA_OK;
}

int mla_decode_stage1(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
                      const int32_t* kv_indices, void* out, float sm_scale, int dtype_mode, mla_plan* workspace,
                      void* stream) {
  int rc = validate_decode(q, kv, kv_scale, kv_indptr, kv_indices, out, dtype_mode, workspace, kRows);
  if (rc != MLA_OK) return rc;
  const mla::DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  return decode_common(a, dtype_mode, workspace, stream, false);
}

int mla_decode_reduce(void* out, mla_plan* workspace, void* stream) {
  if (!workspace || workspace->refcount <= 0) return MLA_ERR_ARG;
  if (workspace->dev.n_reduce == 0) return MLA_OK;
  if (!out) return MLA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 15) return MLA_ERR_ALIGN;
  return mla::launch_reduce(out, workspace->dev, stream, false) == 0 ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
               const int32_t* kv_indices, void* out, float sm_scale, int dtype_mode, mla_plan* workspace,
               void* stream) {
  int rc = validate_decode(q, kv, kv_scale, kv_indptr, kv_indices, out, dtype_mode, workspace, kRows);
  if (rc != MLA_OK) return rc;
  const mla::DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  return decode_common(a, dtype_mode, workspace, stream, true);
}

int mla_decode_paged(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* kv_last_page_len, int page_size, void* out,
                     float sm_scale, int dtype_mode, mla_plan* workspace, void* stream) {
  if (page_size < 1) return MLA_ERR_ARG;
  const Layout l{kPagedKind, page_size, page_size > 1 ? kv_last_page_len : nullptr, nullptr, false};
  int rc = validate_decode(q, kv, kv_scale, kv_indptr, kv_indices, out, dtype_mode, workspace, l);
  if (rc != MLA_OK) return rc;
  mla::DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  a.kv_last_page_len = l.last;
  mla::set_page_size(a, page_size);
  return decode_common(a, dtype_mode, workspace, stream, true);
}

int mla_decode_multi(const void* q, const void* kv, const float* kv_scale, const int32_t* qo_indptr,
                     const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                     int page_size, void* out, float sm_scale, int dtype_mode, mla_plan* workspace, void* stream) {
  if (page_size < 1 || !workspace) return MLA_ERR_ARG;
  const Layout l{kMultiKind, page_size, page_size > 1 ? kv_last_page_len : nullptr, qo_indptr, workspace->causal};
  int rc = validate_decode(q, kv, kv_scale, kv_indptr, kv_indices, out, dtype_mode, workspace, l);
  if (rc != MLA_OK) return rc;
  mla::DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  a.kv_last_page_len = l.last;
  mla::set_page_size(a, page_size);
  a.qo_indptr = qo_indptr;
  return decode_common(a, dtype_mode, workspace, stream, true);
}

int mla_plan_check_error(mla_plan* plan, void* stream) {
  if (!plan || plan->refcount <= 0) return MLA_ERR_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  int code = 0;
  if (cudaMemcpy(&code, plan->dev.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MLA_ERR_CUDA;
  if (code != 0 && cudaMemset(plan->dev.err, 0, sizeof(int)) != cudaSuccess) return MLA_ERR_CUDA;
  return code;
}

const char* mla_strerror(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_ARG: return "invalid argument";
    case MLA_ERR_DTYPE: return "unknown dtype_mode";
    case MLA_ERR_PLAN_MISMATCH: return "device kv_indptr (or last page lengths) does not match the plan";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_TIMEOUT: return "a bounded wait in a kernel timed out";
    case MLA_ERR_ALIGN: return "q, kv or out is not 16-byte aligned";
    case MLA_ERR_NOMEM: return "allocation failed";
    case MLA_ERR_INDEX: return "kv_indices entry out of range";
    case MLA_ERR_DEVICE: return "no usable sm_103 device or wrong device for the plan";
    case MLA_ERR_INDPTR:
      return "kv_indptr must start at 0 and be non-decreasing (and last page lengths lie in [1, page_size])";
    case MLA_ERR_NOALLOC_LIMIT:
      return "request exceeds the fixed scratch of mla_decode_noalloc (batch <= 1024, <= 500 partial slots)";
    default: return "unknown status";
  }
}

int mla_version(void) { return 100; }

// Host-only view of the planner (no CUDA call): fills caller arrays with the
// work list the plan would hold. Any output pointer may be NULL to only count.
static int export_host_plan(int rc, mla::HostPlan& h, int32_t* counts4, int32_t* items5, int items_cap,
                            int32_t* work_indptr, int indptr_cap, int32_t* reduce3, int reduce_cap) {
  if (rc != MLA_OK) return rc;
  counts4[0] = h.n_items;
  counts4[1] = h.num_ctas;
  counts4[2] = h.num_slots;
  counts4[3] = h.n_reduce;
  if (items5 && items_cap >= h.n_items)
    for (int i = 0; i < h.n_items; ++i) {
      items5[5 * i + 0] = h.items[i].b;
      items5[5 * i + 1] = h.items[i].t_begin;
      items5[5 * i + 2] = h.items[i].t_end;
      items5[5 * i + 3] = h.items[i].slot;
      items5[5 * i + 4] = h.items[i].seq_len;
    }
  if (work_indptr && indptr_cap >= h.num_ctas + 1)
    std::memcpy(work_indptr, h.work_indptr, sizeof(int32_t) * (size_t)(h.num_ctas + 1));
  if (reduce3 && reduce_cap >= h.n_reduce)
    for (int i = 0; i < h.n_reduce; ++i) {
      reduce3[3 * i + 0] = h.reduce[i].b;
      reduce3[3 * i + 1] = h.reduce[i].slot_begin;
      reduce3[3 * i + 2] = h.reduce[i].n_slots;
    }
  mla::free_host_plan(&h);
  return MLA_OK;
}

int mla_plan_compute_host(int batch, const int32_t* kv_indptr_host, int num_sms, const mla_plan_options* options,
                          int32_t* counts4, int32_t* items5, int items_cap, int32_t* work_indptr, int indptr_cap,
                          int32_t* reduce3, int reduce_cap) {
  try {
    if (!counts4) return MLA_ERR_ARG;
    mla::HostPlan h;
    static const int32_t kZero = 0;
    const int rc = mla::build_host_plan(batch, batch > 0 ? kv_indptr_host : &kZero, num_sms,
                                        mla::resolve_options(options), &h);
    return export_host_plan(rc, h, counts4, items5, items_cap, work_indptr, indptr_cap, reduce3, reduce_cap);
  } catch (...) {
    return MLA_ERR_NOMEM;
  }
}

int mla_plan_compute_host_multi(int batch, const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                                const int32_t* kv_last_page_len_host, int page_size, int causal, int num_sms,
                                const mla_plan_options* options, int32_t* counts4, int32_t* items8, int items_cap,
                                int32_t* work_indptr, int indptr_cap, int32_t* reduce4, int reduce_cap) {
  try {
    if (!counts4) return MLA_ERR_ARG;
    mla::HostPlan h;
    static const int32_t kZero = 0;
    const int rc = mla::build_host_plan_multi(batch, batch > 0 ? qo_indptr_host : &kZero,
                                              batch > 0 ? kv_indptr_host : &kZero, kv_last_page_len_host, page_size,
                                              causal != 0, num_sms, mla::resolve_options(options), &h);
    if (rc == MLA_OK && items8 && items_cap >= h.n_items)
      for (int i = 0; i < h.n_items; ++i) {
        items8[8 * i + 5] = h.items[i].q_row;
        items8[8 * i + 6] = h.items[i].q_tok;
        items8[8 * i + 7] = h.items[i].pad;
      }
    if (rc == MLA_OK && reduce4 && reduce_cap >= h.n_reduce)
      for (int i = 0; i < h.n_reduce; ++i) reduce4[4 * i + 3] = h.reduce[i].pad;
    // the first five fields of every item at a stride of eight, the first three of every reduce entry at four
    std::vector<int32_t> five(items8 && rc == MLA_OK && items_cap >= h.n_items ? (size_t)h.n_items * 5 : 0);
    std::vector<int32_t> three(reduce4 && rc == MLA_OK && reduce_cap >= h.n_reduce ? (size_t)h.n_reduce * 3 : 0);
    const int n_items = rc == MLA_OK ? h.n_items : 0, n_reduce = rc == MLA_OK ? h.n_reduce : 0;
    const int rc2 = export_host_plan(rc, h, counts4, five.empty() ? nullptr : five.data(), items_cap, work_indptr,
                                     indptr_cap, three.empty() ? nullptr : three.data(), reduce_cap);
    if (rc2 == MLA_OK && !five.empty())
      for (int i = 0; i < n_items; ++i)
        for (int f = 0; f < 5; ++f) items8[8 * i + f] = five[(size_t)i * 5 + f];
    if (rc2 == MLA_OK && !three.empty())
      for (int i = 0; i < n_reduce; ++i)
        for (int f = 0; f < 3; ++f) reduce4[4 * i + f] = three[(size_t)i * 3 + f];
    return rc2;
  } catch (...) {
    return MLA_ERR_NOMEM;
  }
}

int mla_plan_compute_host_paged(int batch, const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                                int page_size, int num_sms, const mla_plan_options* options, int32_t* counts4,
                                int32_t* items5, int items_cap, int32_t* work_indptr, int indptr_cap,
                                int32_t* reduce3, int reduce_cap) {
  try {
    if (!counts4) return MLA_ERR_ARG;
    mla::HostPlan h;
    static const int32_t kZero = 0;
    const int rc = mla::build_host_plan_paged(batch, batch > 0 ? kv_indptr_host : &kZero, kv_last_page_len_host,
                                              page_size, num_sms, mla::resolve_options(options), &h);
    return export_host_plan(rc, h, counts4, items5, items_cap, work_indptr, indptr_cap, reduce3, reduce_cap);
  } catch (...) {
    return MLA_ERR_NOMEM;
  }
}

}  // extern "C"
