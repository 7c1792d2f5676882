// Stage 1 of MLA decode in fp8 mode on the 5th-generation tensor cores of
// sm_103a (tcgen05 + TMEM + TMA). Same work list, outputs and numerics
// contract as the warp-level kernel in stage1.cu; this one exists because the
// legacy warp-level e4m3 mma sustains too little throughput on this GPU for the
// fp8 stream to stay HBM-bound.
//
// Per 128-row KV tile (rows = tokens of one sequence):
//   S^T[128 tokens x 16 heads] = K_tile[128 x 576] . Q^T[576 x 16]
//       tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 16 heads, K = 32 x 18,
//       A = the KV tile (K-major, 128-byte swizzled, straight from TMA),
//       B = the e4m3 query (K-major, 128-byte swizzled), D in TMEM.
//   softmax over tokens per head (4 warps, one thread per token row),
//   P^T written to shared memory as [token][16 heads] e4m3,
//   O^T[512 dims x 16 heads] += V^T[512 x 128] . P^T[128 x 16]
//       four M = 128 MMAs per 32-token k-step, A = the same KV tile read
//       MN-major (dims contiguous), B = P^T MN-major, D in TMEM.
// The value vectors are the first 512 entries of the rows used as keys
// (kernelbot amd-mixed-mla submission 689529 "MLA decode V3", custom_kernel
// passes one KV buffer for both), the query is cast directly to e4m3 with
// scale 1 and the per-tensor kv_scale multiplies the scores and the output
// (submission 690201 "V6c", custom_kernel).
//
// Warp roles (192 threads): warps 0-3 softmax and epilogue (warp w reads TMEM
// lanes 32w..32w+31), warp 4 TMA producer and query staging, warp 5 TMEM
// allocation and the single MMA-issuing thread. Two KV stages of 80 KB,
// double-buffered S, P, Q and O. The running max per head is updated lazily:
// O in TMEM is rescaled only when a tile's max exceeds the reference by more
// than 2^8, so P = 2^(s - m_ref) <= 256 stays inside e4m3's range.
//
// KV rows arrive by TMA: a tile whose 128 row indices are consecutive is
// five 2-D box loads (128 rows x 128 bytes each); any other tile uses 4-row
// gather loads. Rows past the end of an item, and rows whose index is out of
// range, are read at an out-of-bounds coordinate, which TMA fills with zeros.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace mla {
namespace {

constexpr int kRowsU = 128;                 // KV rows per tile = UMMA M of the scores
constexpr int kCB = 5;                      // 128-byte column blocks per row (576 B = 4.5 blocks)
constexpr int kBlk = kRowsU * 128;          // 16 KB per column block
constexpr int kStageU = kCB * kBlk;         // 80 KB per KV stage
constexpr int kQBuf = kCB * 16 * 128;       // 10 KB: e4m3 query, 5 K-blocks x 16 heads x 128 B
constexpr int kPBuf = kRowsU * 16;          // 2 KB: P^T [128 tokens][16 heads] e4m3
constexpr int kThreadsU = 192;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColS = 0;               // S^T: 2 buffers x 16 columns
constexpr uint32_t kColO = 32;              // O^T: 2 buffers x 4 blocks x 16 columns
constexpr float kTau = 8.0f;
constexpr uint64_t kWaitLimitNsU = 2000000000ull;
constexpr uint64_t kDrainLimitNsU = 200000000ull;
constexpr float kLog2eU = 1.4426950408889634f;
constexpr uint32_t kIdescQK = umma::idesc_e4m3(128, 16, 0, 0);
constexpr uint32_t kIdescPV = umma::idesc_e4m3(128, 16, 1, 1);

struct SU {
  static constexpr int kStage = 0;                   // 2 x 80 KB, 1024-aligned
  static constexpr int kQ = 2 * kStageU;             // 2 x 10 KB
  static constexpr int kP = kQ + 2 * kQBuf;          // 2 x 2 KB
  static constexpr int kRed = kP + 2 * kPBuf;        // [2][16 heads][4 warps] fp32 tile max
  static constexpr int kLsum = kRed + 2 * 64 * 4;    // [16 heads][4 warps] fp32 row sums
  static constexpr int kBar = kLsum + 64 * 4;        // 17 mbarriers
  static constexpr int kTmemSlot = kBar + 17 * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kBytes = kAbort + 4;
  static constexpr int kAlloc = kBytes + 1024;       // base is rounded up to 1024 inside the kernel
};
static_assert(SU::kAlloc <= 232448, "tcgen05 stage-1 shared memory");
enum : int {
  kBFull = 0, kBEmpty = 2, kBSFull = 4, kBPFull = 6, kBPEmpty = 8, kBQFull = 10, kBQEmpty = 12, kBOEmpty = 14,
  kBDrain = 16
};

__device__ __forceinline__ void record_error_u(int* err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ bool has_tiles(const WorkItem& w, const int32_t* kv_indptr) {
  return w.t_end > w.t_begin && (int64_t)kv_indptr[w.b + 1] - kv_indptr[w.b] == w.seq_len;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_u(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  while (true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (ptx::globaltimer_ns() - t0 > kWaitLimitNsU) {
      *abort_flag = 1;
      return false;
    }
  }
}

// Tile stream of one CTA (items without rows or with a mismatched length are skipped).
struct TCur {
  int it, it_end;
  int k;          // index of the current item among the items that have tiles
  int t0, t_begin, t_end;
  int b;
  int64_t base;   // kv_indices offset of the sequence's row 0
  bool done;
};
__device__ __forceinline__ void tcur_settle(TCur& c, const DevicePlan& p, const int32_t* ip) {
  while (c.it < c.it_end) {
    const WorkItem w = p.items[c.it];
    if (has_tiles(w, ip)) {
      c.t0 = c.t_begin = w.t_begin;
      c.t_end = w.t_end;
      c.b = w.b;
      c.base = ip[w.b];
      c.done = false;
      return;
    }
    ++c.it;
  }
  c.done = true;
}
__device__ __forceinline__ void tcur_init(TCur& c, int it, int it_end, const DevicePlan& p, const int32_t* ip) {
  c.it = it;
  c.it_end = it_end;
  c.k = 0;
  tcur_settle(c, p, ip);
}
__device__ __forceinline__ void tcur_next(TCur& c, const DevicePlan& p, const int32_t* ip) {
  c.t0 += kRowsU;
  if (c.t0 >= c.t_end) {
    ++c.it;
    ++c.k;
    tcur_settle(c, p, ip);
  }
}

// Warp-wide transpose reduction of 16 per-lane values: returns, in every lane,
// the reduction over the 32 lanes of value (lane >> 1).
template <bool kMax>
__device__ __forceinline__ float xreduce16(const float (&x)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a8[8], a4[4], a2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) a8[i] = op(u16 ? x[i + 8] : x[i], __shfl_xor_sync(~0u, u16 ? x[i] : x[i + 8], 16));
#pragma unroll
  for (int i = 0; i < 4; ++i) a4[i] = op(u8 ? a8[i + 4] : a8[i], __shfl_xor_sync(~0u, u8 ? a8[i] : a8[i + 4], 8));
#pragma unroll
  for (int i = 0; i < 2; ++i) a2[i] = op(u4 ? a4[i + 2] : a4[i], __shfl_xor_sync(~0u, u4 ? a4[i] : a4[i + 2], 4));
  float a1 = op(u2 ? a2[1] : a2[0], __shfl_xor_sync(~0u, u2 ? a2[0] : a2[1], 2));
  return op(a1, __shfl_xor_sync(~0u, a1, 1));
}

__device__ __forceinline__ uint32_t cast4_e4m3(uint32_t bf_lo, uint32_t bf_hi) {
  const float f0 = __uint_as_float(bf_lo << 16), f1 = __uint_as_float(bf_lo & 0xffff0000u);
  const float f2 = __uint_as_float(bf_hi << 16), f3 = __uint_as_float(bf_hi & 0xffff0000u);
  return ptx::f32x2_to_e4m3x2(f0, f1) | (ptx::f32x2_to_e4m3x2(f2, f3) << 16);
}

__global__ void __launch_bounds__(kThreadsU, 1)
    mla_stage1_fp8_umma_kernel(const DecodeArgs a, const DevicePlan p, const __grid_constant__ CUtensorMap tm_tile,
                               const __grid_constant__ CUtensorMap tm_gather, const int32_t oob_row) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((int)blockIdx.x >= p.num_ctas) return;
  const int item_begin = p.work_indptr[blockIdx.x], item_end = p.work_indptr[blockIdx.x + 1];

  // 1024-aligned base for the 128-byte swizzle atoms
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t stage_addr = base + SU::kStage, q_addr = base + SU::kQ, p_addr = base + SU::kP;
  float* red = reinterpret_cast<float*>(smem + SU::kRed);
  float* lsum = reinterpret_cast<float*>(smem + SU::kLsum);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SU::kAbort);
  auto bar = [&](int i) { return base + SU::kBar + 8u * (uint32_t)i; };

  if (tid == 0) {
    ptx::mbar_init(bar(kBFull), 1);
    ptx::mbar_init(bar(kBFull + 1), 1);
    ptx::mbar_init(bar(kBEmpty), 1);
    ptx::mbar_init(bar(kBEmpty + 1), 1);
    ptx::mbar_init(bar(kBSFull), 1);
    ptx::mbar_init(bar(kBSFull + 1), 1);
    ptx::mbar_init(bar(kBPFull), 128);
    ptx::mbar_init(bar(kBPFull + 1), 128);
    ptx::mbar_init(bar(kBPEmpty), 1);
    ptx::mbar_init(bar(kBPEmpty + 1), 1);
    ptx::mbar_init(bar(kBQFull), 32);
    ptx::mbar_init(bar(kBQFull + 1), 32);
    ptx::mbar_init(bar(kBQEmpty), 1);
    ptx::mbar_init(bar(kBQEmpty + 1), 1);
    ptx::mbar_init(bar(kBOEmpty), 128);
    ptx::mbar_init(bar(kBOEmpty + 1), 128);
    ptx::mbar_init(bar(kBDrain), 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 5) {
    umma::tmem_alloc(base + SU::kTmemSlot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + SU::kTmemSlot);
  ptx::griddep_launch_dependents();

  const float kv_scale = __ldg(a.kv_scale);
  const float score_log2 = a.sm_scale * kv_scale * kLog2eU;

  if (warp == 4) {
    // ------------------------------------------------ producer: query staging + KV tiles
    if (lane == 0) {
      umma::tma_prefetch_desc(&tm_tile);
      umma::tma_prefetch_desc(&tm_gather);
    }
    const uint64_t pol = ptx::l2_evict_first_policy();
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
    TCur c;
    tcur_init(c, item_begin, item_end, p, a.kv_indptr);
    int i = 0, q_item = -1;
    bool ok = true;
    while (!c.done && ok) {
      if (c.k != q_item) {  // first tile of an item: stage its e4m3 query (K-major, 128-byte swizzle)
        if (c.k >= 2 && !wait_u(bar(kBQEmpty + (c.k & 1)), ((c.k >> 1) - 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const __nv_bfloat16* qb = q + (int64_t)c.b * kHeads * kQkDim;
        uint8_t* qs = smem + SU::kQ + (c.k & 1) * kQBuf;
        for (int ci = lane; ci < kHeads * 72; ci += 32) {
          const int h = ci / 72, d0 = (ci % 72) * 8;
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qb + h * kQkDim + d0));
          const int kb = d0 >> 7, x = d0 & 127, r = h & 7;
          uint8_t* dst = qs + kb * 2048 + (h >> 3) * 1024 + r * 128 + ((((x >> 4) ^ r)) << 4) + (x & 8);
          *reinterpret_cast<uint2*>(dst) = make_uint2(cast4_e4m3(raw.x, raw.y), cast4_e4m3(raw.z, raw.w));
        }
        umma::fence_proxy_async_smem();
        umma::mbar_arrive(bar(kBQFull + (c.k & 1)));
        q_item = c.k;
      }
      const int s = i & 1;
      if (i >= 2 && !wait_u(bar(kBEmpty + s), ((i >> 1) - 1) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const int nv = min(kRowsU, c.t_end - c.t0);
      int y[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        int v = oob_row;
        if (r < nv) {
          const int idx = __ldg(a.kv_indices + c.base + c.t0 + r);
          if (idx >= 0 && (p.num_kv_slots == 0 || idx < p.num_kv_slots))
            v = idx;
          else
            record_error_u(p.err, MLA_ERR_INDEX);
        }
        y[j] = v;
      }
      const int y0 = __shfl_sync(~0u, y[0], 0);
      bool contiguous = nv == kRowsU && y0 != oob_row;
#pragma unroll
      for (int j = 0; j < 4; ++j) contiguous = contiguous && (y[j] == y0 + lane + 32 * j);
      contiguous = __all_sync(~0u, contiguous);
      const uint32_t fb = bar(kBFull + s), dst = stage_addr + s * kStageU;
      if (lane == 0) ptx::mbar_arrive_expect_tx(fb, kStageU);
      __syncwarp();
      if (contiguous) {
        if (lane < kCB) umma::tma_load_2d(dst + lane * kBlk, &tm_tile, lane * 128, y0, fb, pol);
      } else {
        // lane g gathers rows 4g..4g+3; row r is held by lane (r & 31), slot (r >> 5)
        int ys[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int src = (4 * lane + jj) & 31;
          const int v0 = __shfl_sync(~0u, y[0], src), v1 = __shfl_sync(~0u, y[1], src);
          const int v2 = __shfl_sync(~0u, y[2], src), v3 = __shfl_sync(~0u, y[3], src);
          const int slot = lane >> 3;
          ys[jj] = slot == 0 ? v0 : (slot == 1 ? v1 : (slot == 2 ? v2 : v3));
        }
#pragma unroll
        for (int cb = 0; cb < kCB; ++cb)
          umma::tma_gather4(dst + cb * kBlk + lane * 512, &tm_gather, cb * 128, ys[0], ys[1], ys[2], ys[3], fb, pol);
      }
      ++i;
      tcur_next(c, p, a.kv_indptr);
    }
    if (!ok && lane == 0) record_error_u(p.err, MLA_ERR_TIMEOUT);
    // let issued loads land before the CTA can exit (they already have in the normal path)
    for (int t = (i >= 2 ? i - 2 : 0); t < i; ++t) {
      const uint32_t b_ = bar(kBFull + (t & 1));
      if (ptx::mbar_try_wait(b_, (t >> 1) & 1)) continue;
      (void)ptx::mbar_wait_bounded(b_, (t >> 1) & 1, kDrainLimitNsU);
    }
  } else if (warp == 5) {
    // ------------------------------------------------ MMA issue (one thread)
    if (lane == 0) {
      bool ok = true;
      auto issue_qk = [&](const TCur& c, int i) -> bool {
        const int s = i & 1;
        if (c.t0 == c.t_begin && !wait_u(bar(kBQFull + (c.k & 1)), (c.k >> 1) & 1, abort_flag)) return false;
        if (!wait_u(bar(kBFull + s), (i >> 1) & 1, abort_flag)) return false;
        umma::fence_after_sync();
        const uint32_t a0 = stage_addr + s * kStageU, b0 = q_addr + (c.k & 1) * kQBuf;
        const uint32_t d = tmem + kColS + 16u * (uint32_t)(i & 1);
#pragma unroll
        for (int st = 0; st < 18; ++st) {
          const uint32_t kb = st >> 2, ko = (st & 3) * 32;
          umma::mma_f8f6f4(d, umma::smem_desc(a0 + kb * kBlk + ko, 16, 1024, umma::kLayoutSw128),
                           umma::smem_desc(b0 + kb * 2048 + ko, 16, 1024, umma::kLayoutSw128), kIdescQK, st > 0);
        }
        umma::commit(bar(kBSFull + (i & 1)));
        return true;
      };
      auto issue_pv = [&](const TCur& d, int i) -> bool {
        const int s = i & 1;
        if (!wait_u(bar(kBPFull + (i & 1)), (i >> 1) & 1, abort_flag)) return false;
        const bool first = d.t0 == d.t_begin;
        if (first && d.k >= 2 && !wait_u(bar(kBOEmpty + (d.k & 1)), ((d.k >> 1) - 1) & 1, abort_flag)) return false;
        umma::fence_after_sync();
        const uint32_t a0 = stage_addr + s * kStageU, p0 = p_addr + (i & 1) * kPBuf;
        const uint32_t ob = tmem + kColO + 64u * (uint32_t)(d.k & 1);
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            umma::mma_f8f6f4(ob + 16u * blk, umma::smem_desc(a0 + blk * kBlk + j * 4096, kBlk, 1024, umma::kLayoutSw128),
                             umma::smem_desc(p0 + j * 512, 128, 256, umma::kLayoutNone), kIdescPV,
                             (first && j == 0) ? 0u : 1u);
        umma::commit(bar(kBPEmpty + (i & 1)));
        umma::commit(bar(kBEmpty + s));
        if (d.t0 + kRowsU >= d.t_end) umma::commit(bar(kBQEmpty + (d.k & 1)));
        return true;
      };
      TCur c, d;
      tcur_init(c, item_begin, item_end, p, a.kv_indptr);
      d = c;
      if (!c.done) {
        ok = issue_qk(c, 0);
        tcur_next(c, p, a.kv_indptr);
      }
      for (int t = 0; ok && !d.done; ++t) {
        if (!c.done) {
          ok = issue_qk(c, t + 1);
          tcur_next(c, p, a.kv_indptr);
          if (!ok) break;
        }
        ok = issue_pv(d, t);
        tcur_next(d, p, a.kv_indptr);
      }
      if (!ok) record_error_u(p.err, MLA_ERR_TIMEOUT);
      // every MMA issued by this thread completes before TMEM is released
      umma::commit(bar(kBDrain));
      (void)ptx::mbar_wait_bounded(bar(kBDrain), 0, kDrainLimitNsU);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 0-3, thread = token row)
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int row = 32 * warp + lane;
    int i = 0, k = 0;
    bool aborted = false;
    for (int it = item_begin; it < item_end && !aborted; ++it) {
      const WorkItem w = p.items[it];
      if ((int64_t)a.kv_indptr[w.b + 1] - a.kv_indptr[w.b] != w.seq_len) {
        if (tid == 0) record_error_u(p.err, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      if (w.t_end <= w.t_begin) {  // empty sequence: zeros
        if (w.slot < 0) {
          __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + (int64_t)w.b * kHeads * kVDim;
          for (int e = tid; e < kHeads * kVDim / 8; e += 128) reinterpret_cast<uint4*>(ob)[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      float m_ref[16], l[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m_ref[h] = -INFINITY;
        l[h] = 0.f;
      }
      for (int t0 = w.t_begin; t0 < w.t_end; t0 += kRowsU, ++i) {
        const int nv = min(kRowsU, w.t_end - t0);
        // tcgen05.ld is warp-collective: the warp takes the branch together
        bool ok = __all_sync(~0u, wait_u(bar(kBSFull + (i & 1)), (i >> 1) & 1, abort_flag));
        float x[16];
        if (ok) {
          umma::fence_after_sync();
          umma::tmem_ld16(tmem + lane_off + kColS + 16u * (uint32_t)(i & 1), x);
        }
#pragma unroll
        for (int h = 0; h < 16; ++h) x[h] = (ok && row < nv) ? x[h] * score_log2 : -INFINITY;
        const float mh = xreduce16<true>(x, lane);
        float* rb = red + (i & 1) * 64;
        if (!(lane & 1)) rb[(lane >> 1) * 4 + warp] = mh;
        if (ptx::named_bar_or(1, 128, !ok)) {
          aborted = true;
          break;
        }
        float tmax[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float4 v = *reinterpret_cast<const float4*>(rb + 4 * h);
          tmax[h] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
        }
        if (t0 == w.t_begin) {
#pragma unroll
          for (int h = 0; h < 16; ++h) m_ref[h] = tmax[h];
        } else {
          bool need = false;
#pragma unroll
          for (int h = 0; h < 16; ++h) need |= tmax[h] > m_ref[h] + kTau;
          if (need) {  // rare: move the reference up and rescale O (after P.V of the previous tile lands)
            float alpha[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              const float mn = fmaxf(m_ref[h], tmax[h]);
              alpha[h] = ptx::ex2(m_ref[h] - mn);
              m_ref[h] = mn;
              l[h] *= alpha[h];
            }
            const int pt = i - 1;
            if (__all_sync(~0u, wait_u(bar(kBPEmpty + (pt & 1)), (pt >> 1) & 1, abort_flag))) {
              umma::fence_after_sync();
              const uint32_t ob = tmem + lane_off + kColO + 64u * (uint32_t)(k & 1);
#pragma unroll
              for (int blk = 0; blk < 4; ++blk) {
                float o[16];
                umma::tmem_ld16(ob + 16u * blk, o);
#pragma unroll
                for (int h = 0; h < 16; ++h) o[h] *= alpha[h];
                umma::tmem_st16(ob + 16u * blk, o);
              }
              umma::tmem_wait_st();
            } else {
              ok = false;
            }
          }
        }
        uint32_t pk[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p0 = ptx::ex2(x[4 * j] - m_ref[4 * j]), p1 = ptx::ex2(x[4 * j + 1] - m_ref[4 * j + 1]);
          const float p2 = ptx::ex2(x[4 * j + 2] - m_ref[4 * j + 2]), p3 = ptx::ex2(x[4 * j + 3] - m_ref[4 * j + 3]);
          pk[j] = ptx::f32x2_to_e4m3x2(p0, p1) | (ptx::f32x2_to_e4m3x2(p2, p3) << 16);
          const uint32_t h01 = ptx::e4m3x2_to_f16x2(pk[j] & 0xffffu), h23 = ptx::e4m3x2_to_f16x2(pk[j] >> 16);
          const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
          const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
          l[4 * j] += f01.x;
          l[4 * j + 1] += f01.y;
          l[4 * j + 2] += f23.x;
          l[4 * j + 3] += f23.y;
        }
        if (ok && i >= 2) ok = wait_u(bar(kBPEmpty + (i & 1)), ((i >> 1) - 1) & 1, abort_flag);
        if (ok)
          *reinterpret_cast<uint4*>(smem + SU::kP + (i & 1) * kPBuf + row * 16) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        umma::fence_proxy_async_smem();
        umma::fence_before_sync();
        umma::mbar_arrive(bar(kBPFull + (i & 1)));
      }
      if (aborted) break;

      // -------- epilogue of the item
      const float lh = xreduce16<false>(l, lane);
      if (!(lane & 1)) lsum[(lane >> 1) * 4 + warp] = lh;
      const int tl = i - 1;
      bool ok = wait_u(bar(kBPEmpty + (tl & 1)), (tl >> 1) & 1, abort_flag);
      if (ptx::named_bar_or(1, 128, !ok)) {
        aborted = true;
        break;
      }
      float inv[16], L[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const float4 v = *reinterpret_cast<const float4*>(lsum + 4 * h);
        L[h] = (v.x + v.y) + (v.z + v.w);
        inv[h] = L[h] > 0.f ? kv_scale / L[h] : 0.f;
      }
      umma::fence_after_sync();
      const uint32_t ob = tmem + lane_off + kColO + 64u * (uint32_t)(k & 1);
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        float o[16];
        umma::tmem_ld16(ob + 16u * blk, o);
        const int dcol = 128 * blk + row;
        if (w.slot < 0) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)w.b * kHeads * kVDim + dcol;
#pragma unroll
          for (int h = 0; h < 16; ++h) out[h * kVDim] = __float2bfloat16_rn(o[h] * inv[h]);
        } else {
          float* po = p.part_o + (int64_t)w.slot * kHeads * kVDim + dcol;
#pragma unroll
          for (int h = 0; h < 16; ++h) po[h * kVDim] = o[h] * inv[h];
        }
      }
      if (w.slot >= 0 && tid == 0) {
        float* pl = p.part_lse + (int64_t)w.slot * kHeads;
#pragma unroll
        for (int h = 0; h < 16; ++h) pl[h] = L[h] > 0.f ? m_ref[h] + __log2f(L[h]) : -INFINITY;
      }
      umma::fence_before_sync();
      umma::mbar_arrive(bar(kBOEmpty + (k & 1)));
      ++k;
    }
    if (aborted && tid == 0) record_error_u(p.err, MLA_ERR_TIMEOUT);
  }

  umma::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

int make_kv_maps(const void* kv, int64_t rows, CUtensorMap* tile, CUtensorMap* gather) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return (int)cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kQkDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kQkDim};
  const cuuint32_t box_t[2] = {128, (cuuint32_t)kRowsU}, box_g[2] = {128, 1}, es[2] = {1, 1};
  void* ptr = const_cast<void*>(kv);
  if (enc(tile, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box_t, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS ||
      enc(gather, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box_g, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS)
    return (int)cudaErrorInvalidValue;
  return 0;
}

}  // namespace

int launch_stage1_fp8_umma(const DecodeArgs& a, const DevicePlan& p, void* stream) {
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(mla_stage1_fp8_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SU::kAlloc);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  if (p.num_ctas <= 0) return 0;
  // rows of the KV pool: the tensor maps' second extent; one past it reads as zeros
  const int64_t rows = (p.num_kv_slots > 0 && p.num_kv_slots < 0x7fffffff) ? p.num_kv_slots : 0x7fffffff;
  thread_local const void* cached_kv = nullptr;
  thread_local int64_t cached_rows = -1;
  thread_local CUtensorMap tm_tile, tm_gather;
  if (cached_kv != a.kv || cached_rows != rows) {
    const int rc = make_kv_maps(a.kv, rows, &tm_tile, &tm_gather);
    if (rc != 0) return rc;
    cached_kv = a.kv;
    cached_rows = rows;
  }
  mla_stage1_fp8_umma_kernel<<<p.num_ctas, kThreadsU, SU::kAlloc, static_cast<cudaStream_t>(stream)>>>(
      a, p, tm_tile, tm_gather, (int32_t)rows);
  return (int)cudaGetLastError();
}

}  // namespace mla
