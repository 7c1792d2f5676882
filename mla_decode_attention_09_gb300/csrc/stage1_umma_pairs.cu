// Stage 1 of MLA decode in fp8 mode for two query tokens of a sequence at
// once (speculative decoding, several query tokens per sequence: the pages'
// qo_indptr / max_seqlen_q, kernelbot amd-mixed-mla submission 690201 "V6c",
// _build_cache, and the causal mask of 689529 "V3"), on the 5th-generation
// tensor cores of sm_103a (tcgen05 + TMEM + TMA).
//
// A work item of a token-pair plan holds query tokens j and j + 1 of one
// sequence: token j + 1 attends to rows [t_begin, t_end) and token j to
// [t_begin, pad) (pad <= t_end: the causal prefix one row shorter, or the
// same rows without causality). Both queries, cast to e4m3 like the fp8
// kernel's, form one 32-row B matrix of the score MMA:
//   [S_j^T | S_{j+1}^T][128 tokens x 32] = K_tile[128 x 576] . [Q_j | Q_{j+1}]^T
// so every KV tile is read from HBM and fed to the tensor cores once for two
// tokens. The softmax keeps a running max and row sum per (token, head) and
// masks each token's rows. Each token's weights are two e4m3 terms (hi + lo),
// as in the fp8 kernel; P.V is one N = 64 MMA per k-step with
// B = [P_hi(j) | P_hi(j+1) | P_lo(j) | P_lo(j+1)] into 64 O columns per 128-dim
// block, and the epilogue adds each token's hi and lo columns. The four blocks
// take 256 of the 512 TMEM columns, so O has one buffer: an item's first P.V
// waits for the epilogue of the item before. (Two N = 32 MMAs per k-step into a
// double-buffered O measured 89.7 against 84.2 us for two tokens, B = 64,
// kv_len = 8192.)
//
// The layout of shared memory is that of the a16w8 kernel's paged instance (stage1_umma_a16.cu):
// the staged query is 18 KB, and a tile's P (8 KB: two terms for two tokens)
// lives in that tile's rope slot, whose rope bytes are dead once the tile's
// scores are done. Only two tiles are then in flight: a tile's rope part waits
// for the P.V of the tile two before. The tile maximum exchange buffer is single (the barrier
// that opens every tile orders its reuse) and doubles as the row-sum buffer of
// the epilogue, behind one more barrier.
//
// It is a separate translation unit from the single-token fp8 kernel: that
// kernel's speed follows its generated code (stage1_umma_a16.cu says more).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace mla {
namespace {

constexpr int kRowsU = 128;                   // KV rows per tile = UMMA M of the scores
constexpr int kBlk = kRowsU * 128;            // 16 KB: one 128-byte column block of a tile
constexpr int kLatStage = 4 * kBlk;           // 64 KB: latent / value part (4 column blocks)
constexpr int kRopeStage = kRowsU * 64;       // 8 KB: rope part (64-byte rows)
constexpr int kLatStages = 3;
// P^T of one tile: [128 tokens][16 heads] e4m3 four times: the rounded P (hi)
// of token j, then of token j + 1, then the rounded remainders P - hi (lo) of
// both. To the P.V MMAs, [hi(j) | hi(j+1)] and [lo(j) | lo(j+1)] are two B
// operands of N = 32 columns whose 16-column groups lie kPTok apart.
constexpr int kPTok = kRowsU * 16;            // 2 KB: one token's term
constexpr int kPLo = 2 * kPTok;               // 4 KB: the lo terms after the hi terms
constexpr int kPBuf = 2 * kPLo;               // 8 KB per tile
constexpr uint32_t kTileTx = kLatStage + kRopeStage;
constexpr int kThreadsU = 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                 // S^T: 2 buffers x 32 columns (token j, token j + 1)
constexpr uint32_t kColO = 256;               // O^T: 4 blocks x 64 columns (hi, lo x token j, j + 1), one buffer
// Lazy max: a tile's max is taken (and O rescaled) only when a score exceeds
// the reference max m_ref by more than kTau (log2 units). P is formed as
// 2^(s - m_ref + kPShift) <= 2^(kTau + kPShift) = 256, inside e4m3's range
// (448); the factor 2^kPShift cancels in O / l and is taken out of the LSE. It
// lifts weights down to 2^-(6 + kPShift) of the reference into e4m3's normal
// range, where the hi + lo pair keeps ~8 significant bits; a sharp softmax
// puts most of its weights a few binades below the max.
constexpr float kTau = 3.0f;
constexpr float kPShift = 5.0f;
static_assert(kTau + kPShift <= 8.0f, "P must stay within e4m3's finite range");
constexpr uint64_t kWaitLimitNsU = 2000000000ull;
constexpr uint64_t kDrainLimitNsU = 200000000ull;
constexpr float kLog2eU = 1.4426950408889634f;
constexpr uint32_t kIdescPV = umma::idesc_e4m3(128, 64, 1, 1);
constexpr uint32_t kLayoutSw64 = 4;

enum : int {
  kBFull = 0,     // [3] tile data landed (TMA tx, and every loader lane's cp.async arrival)
  kBLEmpty = 3,   // [3] latent slot free (P.V done)
  kBREmpty = 6,   // [2] rope slot free (the tile's P.V done: the slot held its P)
  kBSFull = 8,    // [2] S^T ready
  kBPFull = 10,   // [2] P^T written into the rope slot (128 arrivals)
  kBPEmpty = 12,  // [2] P^T consumed (P.V done)
  kBQFull = 14,   // query staged (128 arrivals)
  kBQEmpty = 15,  // query consumed (last scores of the item done)
  kBOEmpty = 16,  // [2] O^T read by the epilogue (128 arrivals); only [0] is used: O has one buffer
  kBDrain = 18,   // every MMA of the CTA done (both issuing threads commit)
  kNumBars = 19
};
constexpr int kBQFullArrivals = 128;

// Two tokens' queries of 16 heads each: a 32-row B matrix. Each tile's P is
// written into its rope slot to make room for it.
constexpr int kRopeStages = 2;
constexpr int kNQ = 32;                           // B rows of the score MMA: token j's heads, then token j+1's
constexpr int kQKBlk = kNQ * 128;                 // one 128-dim K-block of the staged query (4 KB)
constexpr int kQLat = 4 * kQKBlk;                 // latent part, 128-byte swizzle (16 KB)
constexpr int kQBytes = kQLat + kNQ * 64;         // + rope part, 64-byte swizzle (2 KB)
constexpr uint32_t kIdescQK = umma::idesc_e4m3(128, kNQ, 0, 0);

struct SU {
  static constexpr int kLat = 0;                               // 3 x 64 KB
  static constexpr int kRope = kLat + kLatStages * kLatStage;  // 2 x 8 KB: rope part, then the tile's P
  static constexpr int kQ = kRope + kRopeStages * kRopeStage;  // 18 KB
  // [2 tokens][16 heads][4 warps] fp32: a tile's maxima, and an item's row sums in its epilogue
  static constexpr int kRed = kQ + kQBytes;
  static constexpr int kBar = kRed + 2 * 64 * 4;
  static constexpr int kTmemSlot = kBar + kNumBars * 8;
  static constexpr int kAbort = kTmemSlot + 4;
  static constexpr int kRowCopy = kAbort + 4;                  // [3] latent slot holds a row-copied tile
  static constexpr int kBytes = kRowCopy + 3 * 4;
  static constexpr int kAlloc = kBytes;                        // the dynamic base must be 1024-aligned
};
static_assert(SU::kAlloc <= 232448, "token-pair tcgen05 stage-1 shared memory");
static_assert(SU::kQ % 1024 == 0 && SU::kRope % 1024 == 0 && SU::kBar % 8 == 0, "operand alignment");
static_assert(kPBuf <= kRopeStage, "a tile's P fits in its rope slot");

__device__ __forceinline__ void record_error_u(int* err, int code) { atomicCAS(err, 0, code); }

// The item's query rows agree with the device qo_indptr: the first as for
// every item, and the second (of a pair item) within the same sequence.
__device__ __forceinline__ bool pair_query_ok(const DecodeArgs& a, const WorkItem& w) {
  return item_query_ok(a, w) && (w.pad < 0 || a.qo_indptr == nullptr || a.qo_indptr[w.b + 1] >= w.q_row + 2);
}
template <bool kPaged>
__device__ __forceinline__ bool has_tiles(const WorkItem& w, const DecodeArgs& a) {
  return w.t_end > w.t_begin && w.pad >= 0 && device_seq_tokens<kPaged>(a, w.b) == w.seq_len &&
         pair_query_ok(a, w);
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

// Idle bookkeeping of a polling loop: returns false once the loop has made no
// progress for the wait limit, or another role aborted.
struct IdleClock {
  uint64_t since = 0;
  __device__ __forceinline__ void reset() { since = 0; }
  __device__ __forceinline__ bool tick(volatile int* abort_flag) {
    __nanosleep(32);
    const uint64_t now = ptx::globaltimer_ns();
    if (since == 0) since = now;
    if (*abort_flag) return false;
    if (now - since > kWaitLimitNsU) {
      *abort_flag = 1;
      return false;
    }
    return true;
  }
};

// Tile stream of one CTA (items without rows or with a mismatched length are skipped).
struct TCur {
  int it, it_end;
  int k;          // index of the current item among the items that have tiles
  int t0, t_begin, t_end;
  int qrow;       // query / output row of the item
  int64_t base;   // kv_indices offset of the sequence's first entry
  bool done;
};
template <bool kPaged>
__device__ __forceinline__ void tcur_settle(TCur& c, const DevicePlan& p, const DecodeArgs& a) {
  while (c.it < c.it_end) {
    const WorkItem w = p.items[c.it];
    if (has_tiles<kPaged>(w, a)) {
      c.t0 = c.t_begin = w.t_begin;
      c.t_end = w.t_end;
      c.qrow = w.q_row;
      c.base = a.kv_indptr[w.b];
      c.done = false;
      return;
    }
    ++c.it;
  }
  c.done = true;
}
template <bool kPaged>
__device__ __forceinline__ void tcur_init(TCur& c, int it, int it_end, const DevicePlan& p, const DecodeArgs& a) {
  c.it = it;
  c.it_end = it_end;
  c.k = 0;
  tcur_settle<kPaged>(c, p, a);
}
template <bool kPaged>
__device__ __forceinline__ void tcur_next(TCur& c, const DevicePlan& p, const DecodeArgs& a) {
  if (c.done) return;
  c.t0 += kRowsU;
  if (c.t0 >= c.t_end) {
    ++c.it;
    ++c.k;
    tcur_settle<kPaged>(c, p, a);
  }
}
// Move to the first tile of the next item.
template <bool kPaged>
__device__ __forceinline__ void tcur_next_item(TCur& c, const DevicePlan& p, const DecodeArgs& a) {
  if (c.done) return;
  ++c.it;
  ++c.k;
  tcur_settle<kPaged>(c, p, a);
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

// Byte offset of query element (token t of the pair, head h, dims d0..d0+7)
// in the staged query: B-matrix row n = 16 t + h in 8-row groups; latent dims
// in 128-byte-swizzled K-blocks, rope dims in a 64-byte-swizzled block.
__device__ __forceinline__ int q_offset(int t, int h, int d0) {
  const int r = h & 7, grp = 2 * t + (h >> 3);
  if (d0 < 512) {
    const int kb = d0 >> 7, x = d0 & 127;
    return kb * kQKBlk + grp * 1024 + r * 128 + (((x >> 4) ^ r) << 4) + (x & 8);
  }
  const int x = d0 - 512;
  return kQLat + grp * 512 + r * 64 + (((x >> 4) ^ ((r >> 1) & 3)) << 4) + (x & 8);
}

// Four bf16 values (two packed words) cast to e4m3, round to nearest even,
// saturating: the fp8 mode's direct cast of the query (scale 1).
__device__ __forceinline__ uint32_t cast4_e4m3(uint32_t bf_lo, uint32_t bf_hi) {
  const float f0 = __uint_as_float(bf_lo << 16), f1 = __uint_as_float(bf_lo & 0xffff0000u);
  const float f2 = __uint_as_float(bf_hi << 16), f3 = __uint_as_float(bf_hi & 0xffff0000u);
  return ptx::f32x2_to_e4m3x2(f0, f1) | (ptx::f32x2_to_e4m3x2(f2, f3) << 16);
}

struct KvMaps {
  CUtensorMap lat_tile, rope_tile;  // 128-row boxes
  CUtensorMap lat_page, rope_page;  // one-page boxes (page sizes 16..64), else unused
};

// Page sizes whose pages are loaded as one box each: a power of two from 16
// to 64 (half a tile). Boxes must start on a 1024-byte swizzle atom (8 latent
// rows); pages of 8 would work too but measured slower than row copies (80
// small boxes per tile).
__host__ __device__ constexpr bool page_boxes(int page_size) {
  return page_size >= 16 && page_size <= 64 && (page_size & (page_size - 1)) == 0;
}

template <bool kPaged>
__global__ void __launch_bounds__(kThreadsU, 1)
    mla_stage1_fp8_pairs_umma_kernel(const DecodeArgs a, const DevicePlan p, const __grid_constant__ KvMaps tm,
                                 const int32_t oob_row) {
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if ((int)blockIdx.x >= p.num_ctas) return;
  constexpr int kLoaders = 2;  // tiles copied row by row are split between warps 4 and 7

  // 1024-aligned base for the swizzle atoms
  // The swizzle atoms need 1024-aligned buffers and the allocation has no room to
  // round the base up: without an aligned base the CTA touches nothing and stops.
  const uint32_t base = ptx::smem_addr(smem_raw);
  if (base & 1023u) {
    if (threadIdx.x == 0) record_error_u(p.err, MLA_ERR_DEVICE);
    return;
  }
  uint8_t* smem = smem_raw;
  const uint32_t lat_addr = base + SU::kLat, rope_addr = base + SU::kRope, q_addr = base + SU::kQ;
  float* red = reinterpret_cast<float*>(smem + SU::kRed);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SU::kAbort);
  volatile int* row_copy = reinterpret_cast<volatile int*>(smem + SU::kRowCopy);
  auto bar = [&](int i) { return base + SU::kBar + 8u * (uint32_t)i; };

  if (tid == 0) {
    for (int i = 0; i < 3; ++i) {
      ptx::mbar_init(bar(kBFull + i), 1 + 32 * kLoaders);  // producer lane 0 + one cp.async arrival per loader lane
      ptx::mbar_init(bar(kBLEmpty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar(kBREmpty + i), 1);
      ptx::mbar_init(bar(kBSFull + i), 1);
      ptx::mbar_init(bar(kBPFull + i), 128);
      ptx::mbar_init(bar(kBPEmpty + i), 1);
      ptx::mbar_init(bar(kBOEmpty + i), 128);
    }
    ptx::mbar_init(bar(kBQFull), kBQFullArrivals);
    ptx::mbar_init(bar(kBQEmpty), 1);
    ptx::mbar_init(bar(kBDrain), 2);
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
  // The launch allows this grid to start while the previous kernel in the
  // stream finishes: everything above touches only this CTA's shared memory and
  // TMEM. The plan's arrays were written when the plan was made and may be
  // read now; the caller's arrays are read only after that kernel completes.
  // Meanwhile the first item's plan entry, kv_indptr entry and query are
  // prefetched into L2 (a prefetch consumes no data).
  const int item_begin = p.work_indptr[blockIdx.x], item_end = p.work_indptr[blockIdx.x + 1];
  if (warp == 7 && lane == 0 && item_begin < item_end) {
    const WorkItem w0 = p.items[item_begin];
    ptx::prefetch_l2(a.kv_indptr + w0.b);
    ptx::prefetch_l2(a.kv_indptr + w0.b + 1);
    if (kPaged) ptx::prefetch_l2(a.kv_last_page_len + w0.b);
    // single-token calls: query row b of the B rows the plan was made for (a
    // multi-token row is known valid only once qo_indptr has been checked)
    if (a.qo_indptr == nullptr)
      umma::bulk_prefetch_l2(static_cast<const __nv_bfloat16*>(a.q) + (int64_t)w0.q_row * kHeads * kQkDim,
                             kHeads * kQkDim * 2);
  }
  ptx::griddep_wait();

  const float kv_scale = __ldg(a.kv_scale);
  const float score_log2 = a.sm_scale * kv_scale * kLog2eU;

  // MMA issue of one tile (one thread): scores, and P.V
  auto issue_qk = [&](const TCur& c, int i) {
    const uint32_t lat = lat_addr + (i % kLatStages) * kLatStage, rope = rope_addr + (i & 1) * kRopeStage;
    const uint32_t d = tmem + kColS + (uint32_t)kNQ * (uint32_t)(i & 1);
    umma::fence_after_sync();
    // row-copied tile: order the cp.async (generic proxy) writes before the tensor core reads them
    if (row_copy[i % kLatStages]) umma::fence_proxy_async_smem();
#pragma unroll
    for (int st = 0; st < 16; ++st) {
      const uint32_t kb = st >> 2, ko = (st & 3) * 32;
      umma::mma_f8f6f4(d, umma::smem_desc(lat + kb * kBlk + ko, 16, 1024, umma::kLayoutSw128),
                       umma::smem_desc(q_addr + kb * kQKBlk + ko, 16, 1024, umma::kLayoutSw128), kIdescQK, st > 0);
    }
#pragma unroll
    for (int st = 0; st < 2; ++st)
      umma::mma_f8f6f4(d, umma::smem_desc(rope + st * 32, 16, 512, kLayoutSw64),
                       umma::smem_desc(q_addr + kQLat + st * 32, 16, 512, kLayoutSw64), kIdescQK, 1u);
    umma::commit(bar(kBSFull + (i & 1)));  // the rope slot frees only after the tile's P.V (it takes P)
    if (c.t0 + kRowsU >= c.t_end) umma::commit(bar(kBQEmpty));
  };
  auto issue_pv = [&](const TCur& d, int i) {
    const bool first = d.t0 == d.t_begin;
    // P^T of tile i sits in tile i's rope slot
    const uint32_t lat = lat_addr + (i % kLatStages) * kLatStage, p0 = rope_addr + (i & 1) * kRopeStage;
    const uint32_t ob = tmem + kColO;
    umma::fence_after_sync();
    // B = [P_hi(j)^T | P_hi(j+1)^T | P_lo(j)^T | P_lo(j+1)^T], one N = 64 MMA per
    // k-step; MN-major without swizzle: 8-token core matrices 128 B apart along K,
    // the 16-column groups kPTok apart along N
#pragma unroll
    for (int blk = 0; blk < 4; ++blk)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t va = umma::smem_desc(lat + blk * kBlk + j * 4096, kBlk, 1024, umma::kLayoutSw128);
        umma::mma_f8f6f4(ob + 64u * blk, va, umma::smem_desc(p0 + j * 512, 128, kPTok, umma::kLayoutNone), kIdescPV,
                         (first && j == 0) ? 0u : 1u);
      }
    umma::commit(bar(kBPEmpty + (i & 1)));
    umma::commit(bar(kBREmpty + (i & 1)));
    umma::commit(bar(kBLEmpty + i % kLatStages));
  };

  if (warp == 4 || warp == 7) {
    // ------------------------------------------------ loaders: KV tiles
    // Every loader walks the same tile stream and takes the same box / row-copy
    // decision from the same indices. Warp 4 issues the box loads; the row copies
    // of a scattered tile are split among the loaders. Every loader waits
    // for every tile's slot and arrives on every tile's full barrier: the loaders
    // then stay in lockstep with the slot barriers, whose parity waits cannot
    // tell a phase from the one two later.
    const bool main_loader = warp == 4;
    const int g = main_loader ? 0 : 1;  // loader rank
    if (main_loader && lane == 0) {
      umma::tma_prefetch_desc(&tm.lat_tile);
      umma::tma_prefetch_desc(&tm.rope_tile);
      if (kPaged && page_boxes(a.page_size)) {
        umma::tma_prefetch_desc(&tm.lat_page);
        umma::tma_prefetch_desc(&tm.rope_page);
      }
    }
    const uint64_t pol = ptx::l2_evict_first_policy();
    // row sources of one tile held by this lane: tokens lane + 32 j. Index loads run two tiles
    // ahead and are turned into rows and checked only when the tile is issued, so the loads
    // stay in flight meanwhile.
    auto load_rows = [&](const TCur& t, int (&y)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        y[j] = (!t.done && r < t.t_end - t.t0) ? __ldg(a.kv_indices + t.base + token_entry<kPaged>(a, t.t0 + r)) : oob_row;
      }
    };
    // rows past the item, and rows outside [0, pool rows), read as zeros (out-of-bounds coordinate)
    auto check_rows = [&](int t0, int nv, int (&y)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t row = token_row<kPaged>(a, y[j], t0 + lane + 32 * j);
        if (lane + 32 * j >= nv) {
          y[j] = oob_row;
        } else if (y[j] < 0 || row >= oob_row) {
          record_error_u(p.err, MLA_ERR_INDEX);
          y[j] = oob_row;
        } else {
          y[j] = (int)row;
        }
      }
    };
    // c: next tile to load; c1, c2: the two after. Queries are staged by the softmax warps.
    TCur c, c1, c2;
    tcur_init<kPaged>(c, item_begin, item_end, p, a);
    c1 = c;
    tcur_next<kPaged>(c1, p, a);
    c2 = c1;
    tcur_next<kPaged>(c2, p, a);
    int y0s[4], y1s[4];
    load_rows(c, y0s);
    load_rows(c1, y1s);
    int i = 0;
    bool ok = true;
    bool decided = false, cont = false, runs = false;  // box / page-box / row-copy decision for tile c
    int y0 = oob_row;
    // page boxes: lane k < nruns loads page k of the tile, whose first KV row is run_y
    const int run_ps = (kPaged && page_boxes(a.page_size)) ? a.page_size : 0;
    int nruns = 0, run_y = oob_row;
    IdleClock idle;
    while (!c.done) {
      bool progress = false;
      if (!c.done) {
        const int ls = i % kLatStages, rs = i & 1;
        const int nv = c.t_end - c.t0;
        if (!decided) {
          // Box loads when the valid rows are consecutive. A tail tile may then
          // read rows past the item (other rows of the pool, or zeros past its
          // end): only done when the pool size is known, and the softmax zeroes
          // those value rows before P.V reads them.
          check_rows(c.t0, nv, y0s);
          y0 = __shfl_sync(~0u, y0s[0], 0);
          cont = y0 != oob_row && (nv >= kRowsU || p.num_kv_slots > 0);
#pragma unroll
          for (int j = 0; j < 4; ++j) cont = cont && (lane + 32 * j >= nv || y0s[j] == y0 + lane + 32 * j);
          cont = __all_sync(~0u, cont);
          runs = false;
          if constexpr (kPaged) {
            if (!cont && run_ps > 0 && (c.t0 & (run_ps - 1)) == 0) {
              // The tile's pages are whole (a page starts every run_ps rows); the
              // last one may extend past the item, read from the caller's page.
              const int src = (lane * run_ps) & 31, slot = (lane * run_ps) >> 5;
              const int v0 = __shfl_sync(~0u, y0s[0], src), v1 = __shfl_sync(~0u, y0s[1], src);
              const int v2 = __shfl_sync(~0u, y0s[2], src), v3 = __shfl_sync(~0u, y0s[3], src);
              nruns = (min(nv, kRowsU) + run_ps - 1) >> a.page_shift;  // run_ps = 2^page_shift; nv counts the item's rows left
              run_y = lane >= nruns ? oob_row : slot == 0 ? v0 : slot == 1 ? v1 : slot == 2 ? v2 : v3;
              // a page with an out-of-range index takes the row-copy path (zeros)
              runs = __all_sync(~0u, lane >= nruns || run_y != oob_row);
            }
          }
          decided = true;
        }
        bool ready;
        if (main_loader) {  // polls: it also stages queries
          ready = i < kLatStages || ptx::mbar_test_wait(bar(kBLEmpty + ls), ((i / kLatStages) - 1) & 1);
          // the rope slot is free once P.V of the tile two before is done
          ready = ready && (i < 2 || ptx::mbar_test_wait(bar(kBREmpty + rs), ((i >> 1) - 1) & 1));
          ready = __shfl_sync(~0u, ready, 0);
        } else {  // the extra loaders have nothing else to do: a bounded blocking wait
          const bool w_ok =
              (i < kLatStages || wait_u(bar(kBLEmpty + ls), ((i / kLatStages) - 1) & 1, abort_flag)) &&
              (i < 2 || wait_u(bar(kBREmpty + rs), ((i >> 1) - 1) & 1, abort_flag));
          if (!__all_sync(~0u, w_ok)) {
            ok = false;
            break;
          }
          ready = true;
        }
        if (ready) {
          const uint32_t fb = bar(kBFull + ls);
          const uint32_t lat = lat_addr + ls * kLatStage, rope = rope_addr + rs * kRopeStage;
          if (main_loader && lane == 0) row_copy[ls] = (cont || runs) ? 0 : 1;  // published by the arrivals below
          if (runs) {
            if (main_loader) {
              if (lane == 0) ptx::mbar_arrive_expect_tx(fb, (uint32_t)(nruns * run_ps * kQkDim));
              __syncwarp();
              if (lane < nruns) {
#pragma unroll
                for (int cb = 0; cb < 4; ++cb)
                  umma::tma_load_2d(lat + cb * kBlk + lane * run_ps * 128, &tm.lat_page, cb * 128, run_y, fb, pol);
                umma::tma_load_2d(rope + lane * run_ps * 64, &tm.rope_page, 512, run_y, fb, pol);
              }
            }
          } else if (cont) {
            if (main_loader) {
              if (lane == 0) ptx::mbar_arrive_expect_tx(fb, kTileTx);
              __syncwarp();
              if (lane < 4) umma::tma_load_2d(lat + lane * kBlk, &tm.lat_tile, lane * 128, y0, fb, pol);
              if (lane == 4) umma::tma_load_2d(rope, &tm.rope_tile, 512, y0, fb, pol);
            }
          } else {
            // Row r's index sits in lane (r & 31), slot (r >> 5); loader g of n copies the
            // latent rows r = g mod n and the rope groups i = g mod n. Latent: lane l
            // copies 16-byte chunk l of the row's 512 bytes into column block l / 8 at
            // chunk (l % 8) ^ (r % 8) (the 128-byte swizzle). Rope: 8 rows per
            // instruction, lane l copies chunk l % 4 of row 8i + l / 4 at chunk
            // (l % 4) ^ ((r / 2) % 4) (the 64-byte swizzle).
            const uint8_t* kv8 = static_cast<const uint8_t*>(a.kv);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll 4
              for (int rr = (g + kLoaders - (32 * j) % kLoaders) % kLoaders; rr < 32; rr += kLoaders) {
                const int r = 32 * j + rr;
                const int yr = __shfl_sync(~0u, y0s[j], rr);
                const bool valid = yr != oob_row;
                const uint32_t dst = lat + (lane >> 3) * kBlk + r * 128 + ((((uint32_t)lane & 7u) ^ (r & 7)) << 4);
                umma::cp_async_16(dst, kv8 + (valid ? (int64_t)yr * kQkDim : 0) + 16 * lane, valid ? 16u : 0u, pol);
              }
            }
#pragma unroll
            for (int i8 = 0; i8 < 16; ++i8) {
              if (i8 % kLoaders != g) continue;
              const int r = 8 * i8 + (lane >> 2);
              const int yr = __shfl_sync(~0u, y0s[i8 >> 2], r & 31);
              const bool valid = yr != oob_row;
              const uint32_t dst = rope + r * 64 + ((((uint32_t)lane & 3u) ^ ((r >> 1) & 3)) << 4);
              umma::cp_async_16(dst, kv8 + (valid ? (int64_t)yr * kQkDim : 0) + 512 + 16 * (lane & 3),
                                valid ? 16u : 0u, pol);
            }
            if (main_loader && lane == 0) umma::mbar_arrive(fb);
          }
          umma::cp_async_arrive_noinc(fb);
          // shift the index pipeline: tile i+1's indices are already loaded, request tile i+2's
#pragma unroll
          for (int j = 0; j < 4; ++j) y0s[j] = y1s[j];
          load_rows(c2, y1s);
          c = c1;
          c1 = c2;
          tcur_next<kPaged>(c2, p, a);
          ++i;
          decided = false;
          progress = true;
        }
      }
      if (progress) {
        idle.reset();
      } else if (!idle.tick(abort_flag)) {
        ok = false;
        break;
      }
    }
    if (!ok && lane == 0) record_error_u(p.err, MLA_ERR_TIMEOUT);
    umma::cp_async_wait_all();
    // let issued loads land before the CTA can exit (they already have in the normal path)
    for (int t = (i >= kLatStages ? i - kLatStages : 0); main_loader && t < i; ++t) {
      const uint32_t b_ = bar(kBFull + t % kLatStages);
      const uint32_t par = (uint32_t)(t / kLatStages) & 1u;
      if (ptx::mbar_try_wait(b_, par)) continue;
      (void)ptx::mbar_wait_bounded(b_, par, kDrainLimitNsU);
    }
  } else if (warp == 5) {
    // ------------------------------------------------ score MMAs (one thread)
    // Scores of tile j need the item's query (first tile), the tile's data, and
    // the S buffer: the softmax of tile j - 2 has read it (its P is written).
    if (lane == 0) {
      bool ok = true;
      TCur c;
      tcur_init<kPaged>(c, item_begin, item_end, p, a);
      int nq = 0;
      while (!c.done) {
        ok = (c.t0 != c.t_begin || wait_u(bar(kBQFull), c.k & 1, abort_flag)) &&
             wait_u(bar(kBFull + nq % kLatStages), (nq / kLatStages) & 1, abort_flag) &&
             (nq < 2 || wait_u(bar(kBPFull + (nq & 1)), ((nq - 2) >> 1) & 1, abort_flag));
        if (!ok) break;
        issue_qk(c, nq);
        ++nq;
        tcur_next<kPaged>(c, p, a);
      }
      if (!ok) record_error_u(p.err, MLA_ERR_TIMEOUT);
      // every MMA of both issuing threads completes before TMEM is released
      umma::commit(bar(kBDrain));
      (void)ptx::mbar_wait_bounded(bar(kBDrain), 0, kDrainLimitNsU);
    }
    __syncwarp();
  } else if (warp == 6) {
    // ------------------------------------------------ P.V MMAs (one thread)
    // P.V of tile j needs the softmax's P, and for an item's first tile the O
    // buffer, freed by the epilogue of the item two before.
    if (lane == 0) {
      bool ok = true;
      TCur d;
      tcur_init<kPaged>(d, item_begin, item_end, p, a);
      int npv = 0;
      while (!d.done) {
        const bool first = d.t0 == d.t_begin;
        ok = (!first || d.k < 1 || wait_u(bar(kBOEmpty), (d.k - 1) & 1, abort_flag)) &&
             wait_u(bar(kBPFull + (npv & 1)), (npv >> 1) & 1, abort_flag);
        if (!ok) break;
        issue_pv(d, npv);
        ++npv;
        tcur_next<kPaged>(d, p, a);
      }
      if (!ok) record_error_u(p.err, MLA_ERR_TIMEOUT);
      umma::commit(bar(kBDrain));
    }
    __syncwarp();
  } else {
    // ------------------------------------------------ softmax + epilogue (warps 0-3, thread = token row)
    const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
    const int row = 32 * warp + lane;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(a.q);
    // Stage the queries of rows qrow and qrow + 1 (consecutive in q) cast to e4m3:
    // 2 x 16 x 72 chunks of 8 values, 18 per thread, loads all in flight. Every
    // thread fences its stores and arrives on the query barrier.
    auto stage_pair = [&](int qrow) {
      const __nv_bfloat16* qb = qg + (int64_t)qrow * kHeads * kQkDim;
      uint4 raw[18];
#pragma unroll
      for (int u = 0; u < 18; ++u) {
        const int ci = tid + 128 * u;  // chunk ci: row ci / 72 of the pair's 32 (token, head) rows
        raw[u] = __ldg(reinterpret_cast<const uint4*>(qb + (ci / 72) * kQkDim + (ci % 72) * 8));
      }
#pragma unroll
      for (int u = 0; u < 18; ++u) {
        const int ci = tid + 128 * u, n = ci / 72, d0 = (ci % 72) * 8;
        *reinterpret_cast<uint2*>(smem + SU::kQ + q_offset(n >> 4, n & 15, d0)) =
            make_uint2(cast4_e4m3(raw[u].x, raw[u].y), cast4_e4m3(raw[u].z, raw[u].w));
      }
      umma::fence_proxy_async_smem();
      umma::mbar_arrive(bar(kBQFull));
    };
    {
      // Queries of the first item with tiles: 128 threads with eighteen 16-byte loads
      // each, all in flight at once, so they land about when the first KV tile does.
      TCur c0;
      tcur_init<kPaged>(c0, item_begin, item_end, p, a);
      if (!c0.done) stage_pair(c0.qrow);
    }
    const float cs = score_log2;  // score (raw units) -> base-2 exponent
    int i = 0, k = 0;
    bool aborted = false;
    for (int it = item_begin; it < item_end && !aborted; ++it) {
      const WorkItem w = p.items[it];
      if (device_seq_tokens<kPaged>(a, w.b) != w.seq_len || !pair_query_ok(a, w)) {
        if (tid == 0) record_error_u(p.err, MLA_ERR_PLAN_MISMATCH);
        continue;
      }
      if (w.t_end <= w.t_begin || w.pad < 0) {  // no KV rows: zeros for the item's one or two rows
        if (w.slot < 0) {
          __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + (int64_t)w.q_row * kHeads * kVDim;
          const int n = (w.pad < 0 ? 1 : 2) * kHeads * kVDim / 8;
          for (int e = tid; e < n; e += 128) reinterpret_cast<uint4*>(ob)[e] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // the next item with tiles, whose queries this item stages at its end
      int next_q = -1;
      for (int jt = it + 1; jt < item_end; ++jt) {
        const WorkItem wn = p.items[jt];
        if (has_tiles<kPaged>(wn, a)) {
          next_q = wn.q_row;
          break;
        }
      }
      // m0 / m1: the reference max per head of token j / j+1 in log2 units, less
      // kPShift, so that a row's weight is P = 2^(x - m) with x the score in log2 units
      float m0[16], m1[16], l0[16], l1[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m0[h] = m1[h] = -INFINITY;
        l0[h] = l1[h] = 0.f;
      }
      for (int t0 = w.t_begin; t0 < w.t_end; t0 += kRowsU, ++i) {
        const int nv = min(kRowsU, w.t_end - t0);  // token j+1's rows in this tile
        const int nv0 = max(0, min(kRowsU, w.pad - t0));  // token j's rows
        const bool stage_next = next_q >= 0 && t0 + kRowsU >= w.t_end;
        if (stage_next && tid == 0) {  // the next queries come from L2 when they are staged
          umma::bulk_prefetch_l2(qg + (int64_t)next_q * kHeads * kQkDim, kHeads * kQkDim * 2);
          umma::bulk_prefetch_l2(qg + (int64_t)(next_q + 1) * kHeads * kQkDim, kHeads * kQkDim * 2);
        }
        // tcgen05.ld is warp-collective: the warp takes the branch together
        bool ok = __all_sync(~0u, wait_u(bar(kBSFull + (i & 1)), (i >> 1) & 1, abort_flag));
        float s0[16], s1[16];  // raw scores (q8 . k8) of this row for the 16 heads of each token
        if (ok) {
          umma::fence_after_sync();
          const uint32_t sc = tmem + lane_off + kColS + (uint32_t)kNQ * (uint32_t)(i & 1);
          umma::tmem_ld16(sc, s0);
          umma::tmem_ld16(sc + 16u, s1);
        }
        const bool v0 = ok && row < nv0, v1 = ok && row < nv;
        // Fast path: every weight at most 2^(kTau + kPShift) needs no tile max
        // (one barrier ORs the check). A timed-out wait also takes the full
        // path, whose barrier then stops every thread.
        const bool first = t0 == w.t_begin;
        bool local_need = first || !ok;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          local_need |= v0 && fmaf(s0[h], cs, -m0[h]) > kTau + kPShift;
          local_need |= v1 && fmaf(s1[h], cs, -m1[h]) > kTau + kPShift;
        }
        if (ptx::named_bar_or(1, 128, local_need)) {
          {
            float x[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) x[h] = v0 ? s0[h] * cs : -INFINITY;
            const float mh = xreduce16<true>(x, lane);
            if (!(lane & 1)) red[(lane >> 1) * 4 + warp] = mh;
          }
          {
            float x[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) x[h] = v1 ? s1[h] * cs : -INFINITY;
            const float mh = xreduce16<true>(x, lane);
            if (!(lane & 1)) red[64 + (lane >> 1) * 4 + warp] = mh;
          }
          if (ptx::named_bar_or(1, 128, !ok)) {
            aborted = true;
            break;
          }
          // New references; alpha = 2^(old - new) rescales what was summed. A token
          // without rows so far keeps m = -inf (its sums are zero: alpha 1).
          float al0[16], al1[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float4 u0 = *reinterpret_cast<const float4*>(red + 4 * h);
            const float4 u1 = *reinterpret_cast<const float4*>(red + 64 + 4 * h);
            const float n0 = fmaxf(m0[h], fmaxf(fmaxf(u0.x, u0.y), fmaxf(u0.z, u0.w)) - kPShift);
            const float n1 = fmaxf(m1[h], fmaxf(fmaxf(u1.x, u1.y), fmaxf(u1.z, u1.w)) - kPShift);
            al0[h] = n0 == -INFINITY ? 1.f : ptx::ex2(m0[h] - n0);
            al1[h] = n1 == -INFINITY ? 1.f : ptx::ex2(m1[h] - n1);
            m0[h] = n0;
            m1[h] = n1;
            l0[h] *= al0[h];
            l1[h] *= al1[h];
          }
          if (!first) {  // move the references up: rescale O once P.V of the previous tile has landed
            const int pt = i - 1;
            if (__all_sync(~0u, wait_u(bar(kBPEmpty + (pt & 1)), (pt >> 1) & 1, abort_flag))) {
              umma::fence_after_sync();
              const uint32_t ob = tmem + lane_off + kColO;
              // kept as a loop (rare path; code layout)
#pragma unroll 1
              for (int blk = 0; blk < 4; ++blk) {
                float o0[16], o1[16];
                umma::tmem_ld16(ob + 64u * blk, o0);
                umma::tmem_ld16(ob + 64u * blk + 16u, o1);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                  o0[h] *= al0[h];
                  o1[h] *= al1[h];
                }
                umma::tmem_st16(ob + 64u * blk, o0);
                umma::tmem_st16(ob + 64u * blk + 16u, o1);
                // the lo columns of both tokens
                umma::tmem_ld16(ob + 64u * blk + 32u, o0);
                umma::tmem_ld16(ob + 64u * blk + 48u, o1);
#pragma unroll
                for (int h = 0; h < 16; ++h) {
                  o0[h] *= al0[h];
                  o1[h] *= al1[h];
                }
                umma::tmem_st16(ob + 64u * blk + 32u, o0);
                umma::tmem_st16(ob + 64u * blk + 48u, o1);
              }
              umma::tmem_wait_st();
            } else {
              ok = false;
            }
          }
        }
        // P = hi + lo in two e4m3 terms per token. hi is P rounded to 4
        // significant bits in f32 (add half a unit of the 4th bit, clear the bits
        // below), which e4m3 holds exactly in its normal range; lo = P - hi is
        // exact in f32 and rounded to e4m3 (4 more significant bits). l sums P
        // itself. A row outside a token's range has weight 0.
        uint32_t pk0[4], pq0[4], pk1[4], pq1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float p0v[4], h0v[4], p1v[4], h1v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = 4 * j + e;
            p0v[e] = v0 ? ptx::ex2(fmaf(s0[h], cs, -m0[h])) : 0.f;
            p1v[e] = v1 ? ptx::ex2(fmaf(s1[h], cs, -m1[h])) : 0.f;
            h0v[e] = __uint_as_float((__float_as_uint(p0v[e]) + 0x00080000u) & 0xfff00000u);
            h1v[e] = __uint_as_float((__float_as_uint(p1v[e]) + 0x00080000u) & 0xfff00000u);
            l0[h] += p0v[e];
            l1[h] += p1v[e];
          }
          pk0[j] = ptx::f32x2_to_e4m3x2(h0v[0], h0v[1]) | (ptx::f32x2_to_e4m3x2(h0v[2], h0v[3]) << 16);
          pq0[j] = ptx::f32x2_to_e4m3x2(p0v[0] - h0v[0], p0v[1] - h0v[1]) |
                   (ptx::f32x2_to_e4m3x2(p0v[2] - h0v[2], p0v[3] - h0v[3]) << 16);
          pk1[j] = ptx::f32x2_to_e4m3x2(h1v[0], h1v[1]) | (ptx::f32x2_to_e4m3x2(h1v[2], h1v[3]) << 16);
          pq1[j] = ptx::f32x2_to_e4m3x2(p1v[0] - h1v[0], p1v[1] - h1v[1]) |
                   (ptx::f32x2_to_e4m3x2(p1v[2] - h1v[2], p1v[3] - h1v[3]) << 16);
        }
        if (ok && row >= nv) {  // row past the item: its value row may hold anything; P.V must see zeros
          uint8_t* vrow = smem + SU::kLat + (i % kLatStages) * kLatStage + row * 128;
#pragma unroll
          for (int cb = 0; cb < 4; ++cb)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) *reinterpret_cast<uint4*>(vrow + cb * kBlk + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        // P goes into this tile's rope slot: its scores are done (S was full), and
        // the P.V two tiles before, which used the slot last, has landed
        if (ok && i >= 2) ok = wait_u(bar(kBPEmpty + (i & 1)), ((i >> 1) - 1) & 1, abort_flag);
        if (ok) {
          uint8_t* pb = smem + SU::kRope + (i & 1) * kRopeStage + row * 16;
          *reinterpret_cast<uint4*>(pb) = make_uint4(pk0[0], pk0[1], pk0[2], pk0[3]);
          *reinterpret_cast<uint4*>(pb + kPTok) = make_uint4(pk1[0], pk1[1], pk1[2], pk1[3]);
          *reinterpret_cast<uint4*>(pb + kPLo) = make_uint4(pq0[0], pq0[1], pq0[2], pq0[3]);
          *reinterpret_cast<uint4*>(pb + kPLo + kPTok) = make_uint4(pq1[0], pq1[1], pq1[2], pq1[3]);
        }
        umma::fence_proxy_async_smem();
        umma::fence_before_sync();
        umma::mbar_arrive(bar(kBPFull + (i & 1)));
        // this item's last scores are done (S was full), so the query buffer is
        // free: stage the next item's queries now
        if (stage_next) stage_pair(next_q);
      }
      if (aborted) break;

      // -------- epilogue of the item
      const float lh0 = xreduce16<false>(l0, lane), lh1 = xreduce16<false>(l1, lane);
      const int tl = i - 1;
      bool ok = wait_u(bar(kBPEmpty + (tl & 1)), (tl >> 1) & 1, abort_flag);
      // every thread is past its last read of the tile maxima, which share the buffer
      if (ptx::named_bar_or(1, 128, !ok)) {
        aborted = true;
        break;
      }
      if (!(lane & 1)) {
        red[(lane >> 1) * 4 + warp] = lh0;
        red[64 + (lane >> 1) * 4 + warp] = lh1;
      }
      (void)ptx::named_bar_or(1, 128, false);
      umma::fence_after_sync();
      const uint32_t ob = tmem + lane_off + kColO;
#pragma unroll 1
      for (int t = 0; t < 2; ++t) {  // token j, then token j + 1
        float inv[16];
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float4 v = *reinterpret_cast<const float4*>(red + 64 * t + 4 * h);
          const float L = (v.x + v.y) + (v.z + v.w);
          inv[h] = L > 0.f ? kv_scale / L : 0.f;
        }
#pragma unroll 1
        for (int blk = 0; blk < 4; ++blk) {
          float o[16];
          float o_lo[16];
          umma::tmem_ld16(ob + 64u * blk + 16u * t, o);
          umma::tmem_ld16(ob + 64u * blk + 32u + 16u * t, o_lo);
#pragma unroll
          for (int h = 0; h < 16; ++h) o[h] += o_lo[h];
          const int dcol = 128 * blk + row;
          if (w.slot < 0) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)(w.q_row + t) * kHeads * kVDim + dcol;
#pragma unroll
            for (int h = 0; h < 16; ++h) out[h * kVDim] = __float2bfloat16_rn(o[h] * inv[h]);
          } else {
            float* po = p.part_o + (int64_t)(w.slot + t) * kHeads * kVDim + dcol;
#pragma unroll
            for (int h = 0; h < 16; ++h) po[h * kVDim] = o[h] * inv[h];
          }
        }
      }
      if (w.slot >= 0 && tid == 0) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          float* pl = p.part_lse + (int64_t)(w.slot + t) * kHeads;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float4 v = *reinterpret_cast<const float4*>(red + 64 * t + 4 * h);
            const float L = (v.x + v.y) + (v.z + v.w);
            pl[h] = L > 0.f ? (t ? m1[h] : m0[h]) + __log2f(L) : -INFINITY;
          }
        }
      }
      umma::fence_before_sync();
      umma::mbar_arrive(bar(kBOEmpty));
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

// Two views of the e4m3 KV pool [rows x 576 bytes] as 128-row tiles: the
// latent part in 128-byte boxes (128-byte swizzle) and the rope part in
// 64-byte boxes (64-byte swizzle).
int make_kv_maps(const void* kv, int64_t rows, int page_size, KvMaps* m) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return (int)cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)kQkDim, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kQkDim};
  const cuuint32_t es[2] = {1, 1};
  void* ptr = const_cast<void*>(kv);
  struct View {
    CUtensorMap* map;
    cuuint32_t w, h;
    CUtensorMapSwizzle sw;
  };
  const View views[4] = {{&m->lat_tile, 128, (cuuint32_t)kRowsU, CU_TENSOR_MAP_SWIZZLE_128B},
                         {&m->rope_tile, 64, (cuuint32_t)kRowsU, CU_TENSOR_MAP_SWIZZLE_64B},
                         {&m->lat_page, 128, (cuuint32_t)page_size, CU_TENSOR_MAP_SWIZZLE_128B},
                         {&m->rope_page, 64, (cuuint32_t)page_size, CU_TENSOR_MAP_SWIZZLE_64B}};
  *m = KvMaps{};
  for (const View& v : views) {
    if (v.h != (cuuint32_t)kRowsU && !page_boxes(page_size)) continue;
    const cuuint32_t box[2] = {v.w, v.h};
    if (enc(v.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, ptr, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, v.sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return (int)cudaErrorInvalidValue;
  }
  return 0;
}

}  // namespace

int launch_stage1_fp8_pairs_umma(const DecodeArgs& a, const DevicePlan& p, void* stream) {
  // the shared-memory opt-in, once per device (idempotent; atomic flags)
  static std::atomic<bool> configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    void* const kernels[2] = {reinterpret_cast<void*>(mla_stage1_fp8_pairs_umma_kernel<false>),
                              reinterpret_cast<void*>(mla_stage1_fp8_pairs_umma_kernel<true>)};
    for (void* k : kernels)
      if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SU::kAlloc);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.num_ctas <= 0) return 0;
  // rows of the KV pool: the tensor maps' second extent; one past it reads as zeros
  const int64_t rows = (p.num_kv_slots > 0 && p.num_kv_slots < 0x7fffffff) ? p.num_kv_slots : 0x7fffffff;
  thread_local const void* cached_kv = nullptr;
  thread_local int64_t cached_rows = -1;
  thread_local int cached_ps = -1;
  thread_local KvMaps maps;
  if (cached_kv != a.kv || cached_rows != rows || cached_ps != a.page_size) {
    cached_kv = nullptr;
    const int rc = make_kv_maps(a.kv, rows, a.page_size, &maps);
    if (rc != 0) return rc;
    cached_kv = a.kv;
    cached_rows = rows;
    cached_ps = a.page_size;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_ctas);
  cfg.blockDim = dim3(kThreadsU);
  cfg.dynamicSmemBytes = SU::kAlloc;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int32_t r32 = (int32_t)rows;
  return a.page_size > 1 ? (int)cudaLaunchKernelEx(&cfg, mla_stage1_fp8_pairs_umma_kernel<true>, a, p, maps, r32)
                         : (int)cudaLaunchKernelEx(&cfg, mla_stage1_fp8_pairs_umma_kernel<false>, a, p, maps, r32);
}

}  // namespace mla
