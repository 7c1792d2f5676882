// Split reduce of MLA decode: merges the normalised fp32 partial outputs of a
// sequence that stage 1 processed in several KV chunks (the pages'
// mla_reduce_v1 call after mla_decode_stage1_asm_fwd, kernelbot amd-mixed-mla
// submission 690201 "V6c", custom_kernel). For each head, with base-2
// log-sum-exps lse_s of the chunks, L = log2 sum_s 2^{lse_s} and
// out = sum_s 2^{lse_s - L} O_s, rounded to bf16.
//
// One CTA of 128 threads per (split sequence, head); each thread owns 4 of the
// 512 output dims, so every partial row is read once with 16-byte loads. A row
// of up to kBatch slots takes one L2 round trip: lane j of every warp loads the
// LSE of slot j while every thread loads its 16 bytes of all the partial rows,
// all in flight at once; the max and the sum of 2^(lse - max) then come from
// warp shuffles. Longer rows find the max and the sum with one slot per lane,
// and read the partial rows kBatch slots at a time. Two instances: kBatch = 8
// (about 64 registers, so a large grid of short rows runs in one wave) and
// kBatch = 32 (about 160 registers) for plans with longer rows.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kReduceThreads = kVDim / 4;  // 128

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& v) {
  acc.x = fmaf(w, v.x, acc.x);
  acc.y = fmaf(w, v.y, acc.y);
  acc.z = fmaf(w, v.z, acc.z);
  acc.w = fmaf(w, v.w, acc.w);
}

template <int kBatch>  // partial rows in flight per thread
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
  // the row's slots lie r.pad apart (token pairs interleave theirs), else consecutively
  const int64_t lse_stride = (int64_t)max(r.pad, 1) * kHeads;
  const int64_t kSlotStride = lse_stride * kVDim;
  const float* po = p.part_o + ((int64_t)r.slot_begin * kHeads + h) * kVDim + 4 * threadIdx.x;
  auto warp_max = [](float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(~0u, x, o));
    return x;
  };
  auto warp_sum = [](float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(~0u, x, o);
    return x;
  };
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (n <= kBatch) {
    const float ls = lane < n ? lse[lane * lse_stride] : -INFINITY;
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      v[u] = u < n ? __ldcs(reinterpret_cast<const float4*>(po + u * kSlotStride)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float m = warp_max(ls);  // the same in every warp
    if (m != -INFINITY) {
      const float wl = exp2f(ls - m);  // 0 for the lanes past the row's slots
      const float inv_z = 1.0f / warp_sum(wl);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) fma4(acc, __shfl_sync(~0u, wl, u) * inv_z, v[u]);
    }
  } else {
    float m = -INFINITY;
    for (int s = lane; s < n; s += 32) m = fmaxf(m, lse[s * lse_stride]);
    m = warp_max(m);
    if (m != -INFINITY) {
      float z = 0.f;
      for (int s = lane; s < n; s += 32) z += exp2f(lse[s * lse_stride] - m);
      const float inv_z = 1.0f / warp_sum(z);
      for (int s0 = 0; s0 < n; s0 += kBatch) {
        // lane j holds the weight of slot s0 + j
        const int cnt = min(kBatch, n - s0);
        const float wl = lane < cnt ? exp2f(lse[(s0 + lane) * lse_stride] - m) * inv_z : 0.f;
        float4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          v[u] = u < cnt ? __ldcs(reinterpret_cast<const float4*>(po + (s0 + u) * kSlotStride))
                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) fma4(acc, __shfl_sync(~0u, wl, u), v[u]);
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
  __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
  const cudaError_t err = p.reduce_max_slots > 8 ? cudaLaunchKernelEx(&cfg, mla_reduce_kernel<32>, p, o, pdl ? 1 : 0)
                                                 : cudaLaunchKernelEx(&cfg, mla_reduce_kernel<8>, p, o, pdl ? 1 : 0);
  return (int)err;
}

}  // namespace mla
