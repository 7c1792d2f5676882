// Split reduce of MLA decode: merges the normalised fp32 partial outputs of a
// sequence that stage 1 processed in several KV chunks (the pages'
// mla_reduce_v1 call after mla_decode_stage1_asm_fwd, kernelbot amd-mixed-mla
// submission 690201 "V6c", custom_kernel). For each head, with base-2
// log-sum-exps lse_s of the chunks, L = log2 sum_s 2^{lse_s} and
// out = sum_s 2^{lse_s - L} O_s, rounded to bf16.
//
// One CTA of 128 threads per (split sequence, head); each thread owns 4 of the
// 512 output dims, so every partial row is read once with 16-byte loads. Rows
// of up to eight slots (the usual case) take one round trip: every thread loads
// all their LSEs and its parts of all their partial rows at once. Longer rows
// find the max and the sum of 2^(lse - max) with one slot per lane, and read
// the partial rows eight slots at a time.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kReduceThreads = kVDim / 4;  // 128
constexpr int kUnroll = 8;

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

__global__ void __launch_bounds__(kReduceThreads)
    mla_reduce_kernel(const DevicePlan p, __nv_bfloat16* __restrict__ out, int use_pdl) {
  const int e = blockIdx.x / kHeads, h = blockIdx.x % kHeads;
  // the plan's reduce map was written when the plan was made: read it while stage 1 finishes
  const ReduceEntry r = e < p.n_reduce ? p.reduce[e] : ReduceEntry{0, 0, 0, 0};
  if (use_pdl) ptx::griddep_wait();  // stage 1 of this decode has finished writing the partials
  // the next kernel in the stream may start its prologue; it waits for this grid before touching memory
  ptx::griddep_launch_dependents();
  if (e >= p.n_reduce) return;
  const int lane = threadIdx.x & 31;
  const int n = r.n_slots;
  const float* lse = p.part_lse + (int64_t)r.slot_begin * kHeads + h;
  float m = -INFINITY;
  if (n > kUnroll) {
    for (int s = lane; s < n; s += 32) m = fmaxf(m, lse[(int64_t)s * kHeads]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(~0u, m, o));
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int64_t kSlotStride = (int64_t)kHeads * kVDim;
  const float* po = p.part_o + ((int64_t)r.slot_begin * kHeads + h) * kVDim + 4 * threadIdx.x;
  if (n <= kUnroll) {
    float4 v[kUnroll];
    float ls[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (u < n) {
        ls[u] = lse[(int64_t)u * kHeads];
        v[u] = __ldcs(reinterpret_cast<const float4*>(po + u * kSlotStride));
      } else {
        ls[u] = -INFINITY;
        v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) mx = fmaxf(mx, ls[u]);
    if (mx != -INFINITY) {
      float wt[kUnroll], z = 0.f;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        wt[u] = exp2f(ls[u] - mx);  // 0 for the unused slots
        z += wt[u];
      }
      const float inv_z = 1.0f / z;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) fma4(acc, wt[u] * inv_z, v[u]);
    }
  } else if (m != -INFINITY) {
    float z = 0.f;
    for (int s = lane; s < n; s += 32) z += exp2f(lse[(int64_t)s * kHeads] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(~0u, z, o);
    const float inv_z = 1.0f / z;
    for (int s0 = 0; s0 < n; s0 += 32) {
      // lane j holds the weight of slot s0 + j
      const int cnt = min(32, n - s0);
      const float wl = lane < cnt ? exp2f(lse[(int64_t)(s0 + lane) * kHeads] - m) * inv_z : 0.f;
      int j = 0;
      for (; j + kUnroll <= cnt; j += kUnroll) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = __ldcs(reinterpret_cast<const float4*>(po + (s0 + j + u) * kSlotStride));
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) fma4(acc, __shfl_sync(~0u, wl, j + u), v[u]);
      }
      for (; j < cnt; ++j) {
        const float4 v = __ldcs(reinterpret_cast<const float4*>(po + (s0 + j) * kSlotStride));
        fma4(acc, __shfl_sync(~0u, wl, j), v);
      }
    }
  }
  uint2 packed;
  packed.x = ptx::pack_bf16x2(acc.x, acc.y);
  packed.y = ptx::pack_bf16x2(acc.z, acc.w);
  *reinterpret_cast<uint2*>(out + ((int64_t)r.b * kHeads + h) * kVDim + 4 * threadIdx.x) = packed;
}

}  // namespace

int launch_reduce(void* out, const DevicePlan& p, void* stream, bool pdl) {
  if (p.n_reduce <= 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.n_reduce * kHeads));
  cfg.blockDim = dim3(kReduceThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t err =
      cudaLaunchKernelEx(&cfg, mla_reduce_kernel, p, static_cast<__nv_bfloat16*>(out), pdl ? 1 : 0);
  return (int)err;
}

}  // namespace mla
