// mla_decode_noalloc: the decode for callers that must not allocate device
// memory. The split-KV work list, the reduce map and the fp32 partial results
// live in one file-scope __device__ array of fixed size instead of a plan's
// cudaMalloc'ed block; planning runs on the host into stack arrays. The
// stage-1 and reduce kernels are the same ones mla_decode launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace mla {
namespace {

// ---- fixed limits of the static scratch (16 MiB on every device that loads the library)
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

// The scratch. In host code this name is only a stand-in, never a device
// pointer: the device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  std::once_flag once;
  int status = MLA_ERR_DEVICE;
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: resolve the scratch address and
// clear the zero row (the source of padding rows in stage-1 tiles).
void setup_device(int dev, DeviceSetup* s) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3) {
    s->status = MLA_ERR_DEVICE;
    return;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    s->status = MLA_ERR_CUDA;
    return;
  }
  if (cudaDeviceGetAttribute(&s->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaMemset(static_cast<unsigned char*>(ptr) + kZeroOff, 0, 2048) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    s->status = MLA_ERR_CUDA;
    return;
  }
  s->scratch = static_cast<unsigned char*>(ptr);
  s->status = MLA_OK;
}

// Work list in fixed-capacity arrays (no heap): the same split as the
// regular planner with its default options (128-row granules balanced across
// CTAs, chunks of at least 128 rows, one CTA per SM).
struct FixedPlan {
  WorkItem items[kMaxItems];
  int32_t indptr[kMaxCtas + 1];
  ReduceEntry reduce[kMaxReduce];
  int64_t cuts[kMaxCtas + 1];
  int n_items, n_ctas, n_reduce, n_slots;
};

// Returns MLA_OK, MLA_ERR_INDPTR, or MLA_ERR_NOALLOC_LIMIT when a fixed capacity is exceeded.
int plan_fixed(int batch, const int32_t* ip, int num_sms, FixedPlan* fp) {
  constexpr int64_t G = 128, kMinRows = 128;
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

}  // namespace
}  // namespace mla

extern "C" int mla_decode_noalloc(const void* q, const void* kv, const float* kv_scale,
                                  const int32_t* kv_indptr_host, const int32_t* kv_indptr,
                                  const int32_t* kv_indices, int batch, int64_t num_kv_slots, void* out,
                                  float sm_scale, int dtype_mode, int* status_dev, void* stream) {
  using namespace mla;
  if (dtype_mode != MLA_MODE_BF16 && dtype_mode != MLA_MODE_FP8 && dtype_mode != MLA_MODE_A16W8)
    return MLA_ERR_DTYPE;
  if (batch < 0 || !status_dev || (batch > 0 && (!kv_indptr_host || !q || !kv || !kv_indptr || !out)))
    return MLA_ERR_ARG;
  if (batch > kMaxBatch) return MLA_ERR_NOALLOC_LIMIT;
  if (dtype_mode != MLA_MODE_BF16 && batch > 0 && !kv_scale) return MLA_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(kv) | reinterpret_cast<uintptr_t>(out)) & 15)
    return MLA_ERR_ALIGN;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  DeviceSetup& s = g_setup[dev];
  std::call_once(s.once, setup_device, dev, &s);
  if (s.status != MLA_OK) return s.status;

  FixedPlan fp;  // on the stack: no heap allocation
  if (batch > 0) {
    const int rc = plan_fixed(batch, kv_indptr_host, s.num_sms, &fp);
    if (rc != MLA_OK) return rc;
    if (kv_indptr_host[batch] > 0 && !kv_indices) return MLA_ERR_ARG;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status_dev, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
  if (batch == 0) return MLA_OK;

  // Upload the work list. From pageable (stack) memory these copies return
  // once the source has been staged, so the stack arrays may go out of scope.
  unsigned char* base = s.scratch;
  if (cudaMemcpyAsync(base + kItemsOff, fp.items, sizeof(WorkItem) * (size_t)fp.n_items, cudaMemcpyHostToDevice,
                      st) != cudaSuccess ||
      cudaMemcpyAsync(base + kIndptrOff, fp.indptr, sizeof(int32_t) * (size_t)(fp.n_ctas + 1),
                      cudaMemcpyHostToDevice, st) != cudaSuccess ||
      (fp.n_reduce > 0 && cudaMemcpyAsync(base + kReduceOff, fp.reduce, sizeof(ReduceEntry) * (size_t)fp.n_reduce,
                                          cudaMemcpyHostToDevice, st) != cudaSuccess))
    return MLA_ERR_CUDA;

  DevicePlan p{};
  p.items = reinterpret_cast<const WorkItem*>(base + kItemsOff);
  p.work_indptr = reinterpret_cast<const int32_t*>(base + kIndptrOff);
  p.reduce = reinterpret_cast<const ReduceEntry*>(base + kReduceOff);
  p.part_o = reinterpret_cast<float*>(base + kPartOff);
  p.part_lse = reinterpret_cast<float*>(base + kLseOff);
  p.err = status_dev;
  p.num_kv_slots = num_kv_slots > 0 ? num_kv_slots : 0;
  p.num_ctas = fp.n_ctas;
  p.n_reduce = fp.n_reduce;
  p.dual_issue = 1;
  const DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  if (launch_stage1(dtype_mode, a, p, base + kZeroOff, stream) != 0) return MLA_ERR_CUDA;
  if (launch_reduce(out, p, stream, true) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}
