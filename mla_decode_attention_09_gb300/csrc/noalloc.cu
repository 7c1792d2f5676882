// mla_decode_noalloc: the decode for callers that must not allocate device
// memory. The split-KV work list, the reduce map and the fp32 partial results
// live in one file-scope __device__ array of fixed size instead of a plan's
// cudaMalloc'ed block; planning runs on the host into stack arrays
// (noalloc_plan.h). The stage-1 and reduce kernels are the same ones
// mla_decode launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "noalloc_plan.h"

namespace mla {
namespace {

using namespace noalloc;

// The scratch. In host code this name is only a stand-in, never a device
// pointer: the device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  std::mutex mu;
  std::atomic<bool> ready{false};    // set once the set-up below has succeeded
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];

// With device `dev` current: resolve the scratch address and clear the zero
// row (the source of padding rows in stage-1 tiles).
int setup_device(int dev, DeviceSetup* s) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess || major != 10 ||
      minor != 3) {
    cudaGetLastError();
    return MLA_ERR_DEVICE;
  }
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaMemset(static_cast<unsigned char*>(ptr) + kZeroOff, 0, 2048) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  s->scratch = static_cast<unsigned char*>(ptr);
  s->num_sms = sms;
  return MLA_OK;
}

// The set-up runs until it succeeds once per device; a failed attempt (for
// example a transient error) leaves the device to be set up by a later call.
// It synchronises the device, so it is not attempted while `stream` is being
// captured (MLA_ERR_CUDA), which would invalidate the caller's capture.
int ensure_setup(int dev, cudaStream_t stream, DeviceSetup& s) {
  if (s.ready.load(std::memory_order_acquire)) return MLA_OK;
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ready.load(std::memory_order_relaxed)) return MLA_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return MLA_ERR_CUDA;
  }
  if (cs != cudaStreamCaptureStatusNone) return MLA_ERR_CUDA;
  const int rc = setup_device(dev, &s);
  if (rc == MLA_OK) s.ready.store(true, std::memory_order_release);
  return rc;
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceSetup& s = g_setup[dev];
  const int setup_rc = ensure_setup(dev, st, s);
  if (setup_rc != MLA_OK) return setup_rc;

  FixedPlan fp;  // on the stack (about 93 KB): no heap allocation
  if (batch > 0) {
    const int rc = plan_fixed(batch, kv_indptr_host, s.num_sms, &fp);
    if (rc != MLA_OK) return rc;
    if (kv_indptr_host[batch] > 0 && !kv_indices) return MLA_ERR_ARG;
  }
  if (cudaMemsetAsync(status_dev, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
  if (batch == 0) return MLA_OK;

  // Upload the work list. From pageable (stack) memory the runtime stages the
  // source before these calls return, so the stack arrays may go out of scope;
  // staging can make a call wait until work queued earlier on the stream is done.
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
  p.reduce_max_slots = 0;
  for (int i = 0; i < fp.n_reduce; ++i) p.reduce_max_slots = std::max(p.reduce_max_slots, fp.reduce[i].n_slots);
  p.dual_issue = 1;
  const DecodeArgs a{q, kv, kv_scale, kv_indptr, kv_indices, out, sm_scale};
  if (launch_stage1(dtype_mode, a, p, base + kZeroOff, stream) != 0) return MLA_ERR_CUDA;
  if (launch_reduce(out, p, stream, true) != 0) return MLA_ERR_CUDA;
  return MLA_OK;
}
