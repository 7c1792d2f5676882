// Stage 1 of MLA decode on sm_103a: a persistent kernel, one CTA per SM, that
// walks the CTA's slice of the planner's work list (runs of KV rows of one
// sequence), streams those rows once through a multi-stage shared-memory ring
// filled by bulk asynchronous copies (one cp.async.bulk per gathered row, so
// the page_size = 1 indirection costs no extra pass), and for each 64-row tile
//   scores  S[16 heads x 64 rows] = Q . K^T  (warp-level mma, heads as M = 16)
//   online softmax (running max m, running sum l, fp32, base-2 exponent)
//   O[16 x 512] += P . V                      (warp-level mma)
// then writes either the final bf16 output (sequence handled by one CTA) or a
// normalised fp32 partial O with its log-sum-exp for the reduce kernel.
//
// This is the pages' mla_decode_stage1_asm_fwd step (kernelbot amd-mixed-mla
// submission 690201 "V6c", custom_kernel: stage 1 writes `logits` — partial
// O despite the name — and `attn_lse`, then mla_reduce_v1 merges them).
//
// Work split inside a CTA (8 warps): for the scores, warp w owns rows
// 8w..8w+7 of the tile over all 576 dims, with Q held in registers as mma A
// fragments; for P.V, warp w owns output dims 64w..64w+63 over all 64 rows.
// The per-tile max and P go through shared memory between two named
// barriers. Every warp also issues the bulk copies for its 8 rows of the tile
// that reuses the just-freed stage, with row indices fetched two tiles ahead.
//
// fp8 mode: Q is rounded to e4m3 while it is loaded (the pages' direct cast
// with scale 1) and scores use e4m3 x e4m3 mma. P.V runs as f16 m16n8k16
// mma with P in f16 and every e4m3 value byte converted to f16 exactly (the
// a16w8 path below): an e4m3 P would keep only 4 significant bits of each
// weight, too few for a sharply peaked softmax. The V fragments are
// assembled from 32-bit shared loads with byte permutes.
//
// a16w8 mode (bf16 Q x e4m3 KV, the "a16w8" configuration of kernelbot
// amd-mixed-mla submission 598454 "v12", docstring): f16 m16n8k16 mma. Q is
// converted bf16 -> f16 once per item (exact for 2^-14 <= |q| < 65520,
// saturating beyond), every e4m3 key and value byte converts to f16 exactly,
// and P is f16. Keys keep the e4m3 ring layout: the four bytes one lane gets
// from an 8-row ldmatrix (dims 4c..4c+3 of a 16-dim chunk) become that lane's
// two B registers, so mma-k 2c, 2c+1 <- dims 4c, 4c+1 and mma-k 2c+8, 2c+9 <-
// dims 4c+2, 4c+3, and the Q fragments follow the same order. Values reuse the
// e4m3 V fragments: their four bytes are rows 2c, 2c+1, 2c+8, 2c+9 of a
// 16-row half, which is the natural m16n8k16 k order, so P stays in row order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace mla {
namespace {

constexpr int kTile = 64;  // KV rows per pipeline stage
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // a bounded wait gives up after 2 s
constexpr uint64_t kDrainLimitNs = 200000000ull;   // waiting for copies after a timeout
constexpr float kLog2e = 1.4426950408889634f;

template <int MODE>
struct Cfg;
template <>
struct Cfg<MLA_MODE_BF16> {
  static constexpr int kRowBytes = kQkDim * 2;       // 1152
  static constexpr int kRowStride = kRowBytes + 16;  // 1168: 8-row ldmatrix without bank conflicts
  static constexpr int kStages = 3;
  static constexpr int kPStride = kTile * 2 + 16;    // bf16 P row of one head (144 B)
  static constexpr int kQSteps = kQkDim / 16;        // 36 mma k-steps of Q
};
template <>
struct Cfg<MLA_MODE_FP8> {
  static constexpr int kRowBytes = kQkDim;           // 576
  static constexpr int kRowStride = kRowBytes + 16;  // 592
  static constexpr int kStages = 5;
  static constexpr int kPStride = kTile * 2 + 16;    // f16 P row of one head (144 B)
  static constexpr int kQSteps = kQkDim / 32;        // 18
};
template <>
struct Cfg<MLA_MODE_A16W8> {
  static constexpr int kRowBytes = kQkDim;           // 576: e4m3 rows
  static constexpr int kRowStride = kRowBytes + 16;  // 592
  static constexpr int kStages = 5;
  static constexpr int kPStride = kTile * 2 + 16;    // f16 P row of one head (144 B)
  static constexpr int kQSteps = kQkDim / 16;        // 36 f16 mma k-steps of Q
};

template <int MODE>
struct Smem {
  using C = Cfg<MODE>;
  static constexpr int kStageBytes = kTile * C::kRowStride;
  static constexpr int kPOff = C::kStages * kStageBytes;
  static constexpr int kRedOff = kPOff + 16 * C::kPStride;   // [8 warps][16 heads] fp32 tile max
  static constexpr int kSumOff = kRedOff + kWarps * 16 * 4;  // [2][8 warps][16 heads] fp32 row sums
  static constexpr int kBarOff = kSumOff + 2 * kWarps * 16 * 4;
  static constexpr int kBytes = kBarOff + C::kStages * 8;
};
static_assert(Smem<MLA_MODE_BF16>::kBytes <= 232448, "bf16 stage-1 shared memory");
static_assert(Smem<MLA_MODE_FP8>::kBytes <= 232448, "fp8 stage-1 shared memory");
static_assert(Smem<MLA_MODE_A16W8>::kBytes <= 232448, "a16w8 stage-1 shared memory");

__device__ __forceinline__ void record_error(int* err, int code) { atomicCAS(err, 0, code); }

template <bool kPaged>
__device__ __forceinline__ bool item_has_tiles(const WorkItem& w, const DecodeArgs& a) {
  return w.t_end > w.t_begin && device_seq_tokens<kPaged>(a, w.b) == w.seq_len && item_query_ok(a, w);
}

// Position in a CTA's stream of tiles.
struct Cursor {
  int item, item_end;
  int t, t_end;   // first token of the current tile / end token of the item (relative to the sequence)
  int64_t base;   // kv_indices offset of the sequence's first entry
};

template <bool kPaged>
__device__ __forceinline__ void cursor_settle(Cursor& c, const DevicePlan& p, const DecodeArgs& a) {
  while (c.item < c.item_end) {
    const WorkItem w = p.items[c.item];
    if (item_has_tiles<kPaged>(w, a)) {
      c.t = w.t_begin;
      c.t_end = w.t_end;
      c.base = a.kv_indptr[w.b];
      return;
    }
    ++c.item;
  }
}
template <bool kPaged>
__device__ __forceinline__ void cursor_next(Cursor& c, const DevicePlan& p, const DecodeArgs& a) {
  if (c.item >= c.item_end) return;
  c.t += kTile;
  if (c.t >= c.t_end) {
    ++c.item;
    cursor_settle<kPaged>(c, p, a);
  }
}

// Source of one ring row of a future tile: state 0 = nothing, 1 = the zero
// row (past the end of the item), 2 = token `t` of the sequence, whose
// kv_indices entry (a row, or a page id) is `idx`.
struct RowSrc {
  int state;
  int idx;
  int t;
};

template <bool kPaged>
__device__ __forceinline__ RowSrc prefetch_row(const Cursor& c, int r, const DecodeArgs& a) {
  RowSrc s{0, 0, 0};
  if (c.item >= c.item_end) return s;
  if (c.t + r < c.t_end) {
    s.state = 2;
    s.t = c.t + r;
    s.idx = __ldg(a.kv_indices + c.base + token_entry<kPaged>(a, s.t));
  } else {
    s.state = 1;
  }
  return s;
}

template <int MODE, bool kPaged>
__device__ __forceinline__ void issue_row(const RowSrc& s, uint32_t dst, uint32_t bar, const DecodeArgs& a,
                                          const uint8_t* zero_row, int64_t num_kv_slots, int* err,
                                          uint64_t policy) {
  if (s.state == 0) return;
  const uint8_t* src = zero_row;
  if (s.state == 2) {
    const int64_t row = token_row<kPaged>(a, s.idx, s.t);
    if (s.idx >= 0 && (num_kv_slots == 0 || row < num_kv_slots))
      src = static_cast<const uint8_t*>(a.kv) + row * Cfg<MODE>::kRowBytes;
    else
      record_error(err, MLA_ERR_INDEX);
  }
  ptx::bulk_g2s(dst, src, Cfg<MODE>::kRowBytes, bar, policy);
}

// Q of sequence b as mma A fragments: rows are heads g and g + 8.
template <int MODE>
__device__ __forceinline__ void load_q(uint32_t (&qa)[Cfg<MODE>::kQSteps][4], const __nv_bfloat16* q, int b, int g,
                                       int c) {
  const __nv_bfloat16* q0 = q + ((int64_t)b * kHeads + g) * kQkDim;
  const __nv_bfloat16* q1 = q0 + 8 * kQkDim;
  if constexpr (MODE == MLA_MODE_BF16) {
    // m16n8k16 A: a0 = (g, 2c..2c+1), a1 = (g+8, 2c..), a2 = (g, 2c+8..), a3 = (g+8, 2c+8..)
#pragma unroll
    for (int s = 0; s < Cfg<MODE>::kQSteps; ++s) {
      const int k = 16 * s + 2 * c;
      qa[s][0] = __ldg(reinterpret_cast<const uint32_t*>(q0 + k));
      qa[s][1] = __ldg(reinterpret_cast<const uint32_t*>(q1 + k));
      qa[s][2] = __ldg(reinterpret_cast<const uint32_t*>(q0 + k + 8));
      qa[s][3] = __ldg(reinterpret_cast<const uint32_t*>(q1 + k + 8));
    }
  } else if constexpr (MODE == MLA_MODE_A16W8) {
    // m16n8k16 f16 A in the permuted k order of the scores: a0 = (g, dims 4c, 4c+1),
    // a1 = (g+8, dims 4c, 4c+1), a2 = (g, dims 4c+2, 4c+3), a3 = (g+8, dims 4c+2, 4c+3)
    auto to_f16 = [](uint32_t bf2) -> uint32_t {
      return ptx::pack_f16x2_sat(__uint_as_float(bf2 << 16), __uint_as_float(bf2 & 0xffff0000u));
    };
#pragma unroll
    for (int s = 0; s < Cfg<MODE>::kQSteps; ++s) {
      const int k = 16 * s + 4 * c;
      const uint2 r0 = __ldg(reinterpret_cast<const uint2*>(q0 + k));
      const uint2 r1 = __ldg(reinterpret_cast<const uint2*>(q1 + k));
      qa[s][0] = to_f16(r0.x);
      qa[s][1] = to_f16(r1.x);
      qa[s][2] = to_f16(r0.y);
      qa[s][3] = to_f16(r1.y);
    }
  } else {
    // m16n8k32 e4m3 A: a0 = (g, 4c..4c+3), a1 = (g+8, 4c..), a2 = (g, 4c+16..), a3 = (g+8, 4c+16..)
    auto cast4 = [](const __nv_bfloat16* ptr) -> uint32_t {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(ptr));
      const float f0 = __uint_as_float(raw.x << 16), f1 = __uint_as_float(raw.x & 0xffff0000u);
      const float f2 = __uint_as_float(raw.y << 16), f3 = __uint_as_float(raw.y & 0xffff0000u);
      return ptx::f32x2_to_e4m3x2(f0, f1) | (ptx::f32x2_to_e4m3x2(f2, f3) << 16);
    };
#pragma unroll
    for (int s = 0; s < Cfg<MODE>::kQSteps; ++s) {
      const int k = 32 * s + 4 * c;
      qa[s][0] = cast4(q0 + k);
      qa[s][1] = cast4(q1 + k);
      qa[s][2] = cast4(q0 + k + 16);
      qa[s][3] = cast4(q1 + k + 16);
    }
  }
}

template <int MODE, bool kPaged>
__global__ void __launch_bounds__(kThreads, 1)
    mla_stage1_kernel(const DecodeArgs a, const DevicePlan p, const uint8_t* __restrict__ zero_row) {
  using C = Cfg<MODE>;
  using S = Smem<MODE>;
  extern __shared__ __align__(128) uint8_t smem[];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  if ((int)blockIdx.x >= p.num_ctas) return;

  const uint32_t ring = ptx::smem_addr(smem);
  uint8_t* pbuf = smem + S::kPOff;
  float* red = reinterpret_cast<float*>(smem + S::kRedOff);
  float* lsum = reinterpret_cast<float*>(smem + S::kSumOff);
  const uint32_t bar0 = ptx::smem_addr(smem + S::kBarOff);

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) ptx::mbar_init(bar0 + 8u * s, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  ptx::griddep_launch_dependents();
  // The launch allows this grid to start while the previous kernel in the
  // stream finishes; wait for that kernel's completion before any global access.
  ptx::griddep_wait();
  const int item_begin = p.work_indptr[blockIdx.x], item_end = p.work_indptr[blockIdx.x + 1];

  // Tiles this CTA will process (same skipping rules as the item loop below).
  int n_tiles = 0;
  for (int it = item_begin; it < item_end; ++it) {
    const WorkItem w = p.items[it];
    if (item_has_tiles<kPaged>(w, a)) n_tiles += (w.t_end - w.t_begin + kTile - 1) / kTile;
  }

  const float kv_scale = (MODE != MLA_MODE_BF16) ? __ldg(a.kv_scale) : 1.0f;
  const float score_log2 = a.sm_scale * kv_scale * kLog2e;  // score -> base-2 exponent
  const uint64_t policy = ptx::l2_evict_first_policy();

  // ---- copy issue: lanes 0..7 of warp w copy rows 8w..8w+7 of every tile
  const int my_row = warp * 8 + (lane & 7);
  const bool copier = lane < 8;
  const uint32_t my_dst = ring + my_row * C::kRowStride;
  Cursor pc{item_begin, item_end, 0, 0, 0};
  cursor_settle<kPaged>(pc, p, a);
  const int n_pro = min(C::kStages - 1, n_tiles);
  if (tid == 0)
    for (int k = 0; k < n_pro; ++k) ptx::mbar_arrive_expect_tx(bar0 + 8u * k, kTile * C::kRowBytes);
  __syncthreads();  // barriers initialised, expected bytes registered before any copy lands
  for (int k = 0; k < n_pro; ++k) {
    if (copier) {
      const RowSrc rs = prefetch_row<kPaged>(pc, my_row, a);
      issue_row<MODE, kPaged>(rs, my_dst + k * S::kStageBytes, bar0 + 8u * k, a, zero_row, p.num_kv_slots, p.err, policy);
    }
    cursor_next<kPaged>(pc, p, a);
  }
  // sources of tiles n_pro and n_pro + 1 (issued from the loop once stages free up)
  RowSrc pf1 = copier ? prefetch_row<kPaged>(pc, my_row, a) : RowSrc{0, 0};
  cursor_next<kPaged>(pc, p, a);
  RowSrc pf2 = copier ? prefetch_row<kPaged>(pc, my_row, a) : RowSrc{0, 0};
  cursor_next<kPaged>(pc, p, a);

  // ---- consumer state
  uint32_t qa[C::kQSteps][4];
  float o[8][4];
  float m_run[2], l_run[2];  // heads g and g+8: running max (base 2) and this thread's partial row sum
  bool timed_out = false;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  int tile = 0;
  int parity_item = 0;

  for (int it = item_begin; it < item_end; ++it) {
    const WorkItem w = p.items[it];
    if (device_seq_tokens<kPaged>(a, w.b) != w.seq_len || !item_query_ok(a, w)) {
      if (tid == 0) record_error(p.err, MLA_ERR_PLAN_MISMATCH);
      continue;  // skipped by the copy cursor as well
    }
    const int n_rows = w.t_end - w.t_begin;
    if (n_rows > 0) load_q<MODE>(qa, q, w.q_row, g, c);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    m_run[0] = m_run[1] = -INFINITY;
    l_run[0] = l_run[1] = 0.f;

    for (int t0 = 0; t0 < n_rows; t0 += kTile, ++tile) {
      const int stage = tile % C::kStages;
      const uint32_t sbase = ring + stage * S::kStageBytes;
      const int n_valid = min(kTile, n_rows - t0);
      const bool ok = ptx::mbar_wait_bounded(bar0 + 8u * stage, (uint32_t)(tile / C::kStages) & 1u, kWaitLimitNs);

      // ---------------- scores of rows 8w .. 8w+7
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        // ldmatrix.x4: lane supplies row (lane & 7) of the warp's 8 rows, 16-byte chunk (lane >> 3)
        const uint32_t rowaddr = sbase + (warp * 8 + (lane & 7)) * C::kRowStride + (lane >> 3) * 16;
        if constexpr (MODE == MLA_MODE_BF16) {
#pragma unroll
          for (int s2 = 0; s2 < 18; ++s2) {  // 64 bytes = two k16 steps per ldmatrix.x4
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4(rowaddr + s2 * 64, b0, b1, b2, b3);
            ptx::mma_bf16_16816(sacc, qa[2 * s2], b0, b1);
            ptx::mma_bf16_16816(sacc, qa[2 * s2 + 1], b2, b3);
          }
        } else if constexpr (MODE == MLA_MODE_A16W8) {
#pragma unroll
          for (int s2 = 0; s2 < 9; ++s2) {  // 64 bytes = four 16-dim k steps per ldmatrix.x4
            uint32_t b[4];
            ptx::ldsm_x4(rowaddr + s2 * 64, b[0], b[1], b[2], b[3]);
#pragma unroll
            for (int j = 0; j < 4; ++j)  // b[j]: key bytes of dims 16(4 s2 + j) + 4c .. +3 of row g
              ptx::mma_f16_16816(sacc, qa[4 * s2 + j], ptx::e4m3x2_to_f16x2(b[j] & 0xffffu),
                                 ptx::e4m3x2_to_f16x2(b[j] >> 16));
          }
        } else {
#pragma unroll
          for (int s2 = 0; s2 < 9; ++s2) {  // 64 bytes = two k32 steps per ldmatrix.x4
            uint32_t b0, b1, b2, b3;
            ptx::ldsm_x4(rowaddr + s2 * 64, b0, b1, b2, b3);
            ptx::mma_e4m3_16832(sacc, qa[2 * s2], b0, b1);
            ptx::mma_e4m3_16832(sacc, qa[2 * s2 + 1], b2, b3);
          }
        }
      }
      // sacc = S(head g, rows r0, r0+1), S(head g+8, rows r0, r0+1)
      const int r0 = warp * 8 + 2 * c;
      float x[4];
      x[0] = (r0 < n_valid) ? sacc[0] * score_log2 : -INFINITY;
      x[1] = (r0 + 1 < n_valid) ? sacc[1] * score_log2 : -INFINITY;
      x[2] = (r0 < n_valid) ? sacc[2] * score_log2 : -INFINITY;
      x[3] = (r0 + 1 < n_valid) ? sacc[3] * score_log2 : -INFINITY;
      float mx0 = fmaxf(x[0], x[1]), mx1 = fmaxf(x[2], x[3]);
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      if (c == 0) {
        red[warp * 16 + g] = mx0;
        red[warp * 16 + g + 8] = mx1;
      }
      // Tile tile + kStages - 1 goes into the stage tile - 1 used. Every thread
      // has finished waiting on that stage's previous phase (it passed the
      // second barrier of tile - 1), so its expected bytes can be set now.
      const int ahead = tile + C::kStages - 1;
      const int next_stage = ahead % C::kStages;
      if (tid == 0 && ahead < n_tiles) ptx::mbar_arrive_expect_tx(bar0 + 8u * next_stage, kTile * C::kRowBytes);
      if (ptx::named_bar_or(1, kThreads, !ok)) {  // barrier 1; any thread timed out -> all stop
        timed_out = true;
        break;
      }
      // Barrier 1 also means every warp finished P.V of tile - 1: its stage is free.
      if (copier && ahead < n_tiles)
        issue_row<MODE, kPaged>(pf1, my_dst + next_stage * S::kStageBytes, bar0 + 8u * next_stage, a, zero_row,
                        p.num_kv_slots, p.err, policy);
      pf1 = pf2;
      pf2 = copier ? prefetch_row<kPaged>(pc, my_row, a) : RowSrc{0, 0};
      cursor_next<kPaged>(pc, p, a);

      // ---------------- online softmax over the tile
      float tmax0 = red[g], tmax1 = red[g + 8];
#pragma unroll
      for (int w2 = 1; w2 < kWarps; ++w2) {
        tmax0 = fmaxf(tmax0, red[w2 * 16 + g]);
        tmax1 = fmaxf(tmax1, red[w2 * 16 + g + 8]);
      }
      const float mn0 = fmaxf(m_run[0], tmax0), mn1 = fmaxf(m_run[1], tmax1);
      const float alpha0 = ptx::ex2(m_run[0] - mn0), alpha1 = ptx::ex2(m_run[1] - mn1);
      m_run[0] = mn0;
      m_run[1] = mn1;
      const float p0 = ptx::ex2(x[0] - mn0), p1 = ptx::ex2(x[1] - mn0);
      const float p2 = ptx::ex2(x[2] - mn1), p3 = ptx::ex2(x[3] - mn1);
      float ps01, ps23;  // sums of P as rounded for the mma
      if constexpr (MODE == MLA_MODE_BF16) {
        const uint32_t u01 = ptx::pack_bf16x2(p0, p1), u23 = ptx::pack_bf16x2(p2, p3);
        ps01 = __uint_as_float(u01 << 16) + __uint_as_float(u01 & 0xffff0000u);
        ps23 = __uint_as_float(u23 << 16) + __uint_as_float(u23 & 0xffff0000u);
        *reinterpret_cast<uint32_t*>(pbuf + g * C::kPStride + r0 * 2) = u01;
        *reinterpret_cast<uint32_t*>(pbuf + (g + 8) * C::kPStride + r0 * 2) = u23;
      } else {  // fp8 and a16w8: f16 P (P <= 1 against the exact running max)
        const uint32_t u01 = ptx::pack_f16x2(p0, p1), u23 = ptx::pack_f16x2(p2, p3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&u01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&u23));
        ps01 = f01.x + f01.y;
        ps23 = f23.x + f23.y;
        *reinterpret_cast<uint32_t*>(pbuf + g * C::kPStride + r0 * 2) = u01;
        *reinterpret_cast<uint32_t*>(pbuf + (g + 8) * C::kPStride + r0 * 2) = u23;
      }
      l_run[0] = l_run[0] * alpha0 + ps01;
      l_run[1] = l_run[1] * alpha1 + ps23;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        o[i][0] *= alpha0;
        o[i][1] *= alpha0;
        o[i][2] *= alpha1;
        o[i][3] *= alpha1;
      }
      ptx::named_bar_sync(2, kThreads);  // barrier 2: P visible

      // ---------------- O[:, 64w .. 64w+63] += P . V
      const uint32_t pa_addr =
          ptx::smem_addr(pbuf) + ((lane & 7) + 8 * ((lane >> 3) & 1)) * C::kPStride + (lane >> 4) * 16;
      if constexpr (MODE == MLA_MODE_BF16) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 16 rows per k step
          uint32_t pa[4];
          ptx::ldsm_x4(pa_addr + kk * 32, pa[0], pa[1], pa[2], pa[3]);
          const uint32_t vrow = sbase + (16 * kk + (lane & 7) + 8 * ((lane >> 3) & 1)) * C::kRowStride +
                                (64 * warp + 8 * (lane >> 4)) * 2;
#pragma unroll
          for (int np = 0; np < 4; ++np) {  // two n8 tiles (16 dims) per ldmatrix.x4.trans
            uint32_t v0, v1, v2, v3;
            ptx::ldsm_x4_trans(vrow + np * 32, v0, v1, v2, v3);
            ptx::mma_bf16_16816(o[2 * np], pa, v0, v1);
            ptx::mma_bf16_16816(o[2 * np + 1], pa, v2, v3);
          }
        }
      } else {
        // e4m3 V fragments of 32 rows x 32 dims: bb[h][i] holds rows 16h + 2c, +1, +8, +9 (bytes 0..3)
        // of dim 64w + 32blk + 4g + i
        auto v_frags = [&](int kk, int blk, uint32_t (&bb)[2][4]) {
          const uint32_t a0 = sbase + (32 * kk + 2 * c) * C::kRowStride + 64 * warp + 32 * blk + 4 * g;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t ah = a0 + 16 * h * C::kRowStride;
            const uint32_t w0 = ptx::lds32(ah), w1 = ptx::lds32(ah + C::kRowStride);
            const uint32_t w2 = ptx::lds32(ah + 8 * C::kRowStride), w3 = ptx::lds32(ah + 9 * C::kRowStride);
            const uint32_t t0 = ptx::prmt(w0, w1, 0x5140), t1 = ptx::prmt(w0, w1, 0x7362);
            const uint32_t t2 = ptx::prmt(w2, w3, 0x5140), t3 = ptx::prmt(w2, w3, 0x7362);
            bb[h][0] = ptx::prmt(t0, t2, 0x5410);
            bb[h][1] = ptx::prmt(t0, t2, 0x7632);
            bb[h][2] = ptx::prmt(t1, t3, 0x5410);
            bb[h][3] = ptx::prmt(t1, t3, 0x7632);
          }
        };
        {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {  // 32 rows = two f16 k steps (P in row order)
            uint32_t pa[2][4];
            ptx::ldsm_x4(pa_addr + (2 * kk) * 32, pa[0][0], pa[0][1], pa[0][2], pa[0][3]);
            ptx::ldsm_x4(pa_addr + (2 * kk + 1) * 32, pa[1][0], pa[1][1], pa[1][2], pa[1][3]);
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {  // n-tile i column n = dim 64w + 32blk + 4n + i
              uint32_t bb[2][4];
              v_frags(kk, blk, bb);
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  ptx::mma_f16_16816(o[4 * blk + i], pa[h], ptx::e4m3x2_to_f16x2(bb[h][i] & 0xffffu),
                                     ptx::e4m3x2_to_f16x2(bb[h][i] >> 16));
            }
          }
        }
      }
    }
    if (timed_out) break;

    // ---------------- epilogue: O / l (x kv_scale), final bf16 or partial fp32 + LSE
    float l0 = l_run[0], l1 = l_run[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    float* ls = lsum + parity_item * (kWarps * 16);
    parity_item ^= 1;
    if (c == 0) {
      ls[warp * 16 + g] = l0;
      ls[warp * 16 + g + 8] = l1;
    }
    ptx::named_bar_sync(1, kThreads);
    float L0 = 0.f, L1 = 0.f;
#pragma unroll
    for (int w2 = 0; w2 < kWarps; ++w2) {
      L0 += ls[w2 * 16 + g];
      L1 += ls[w2 * 16 + g + 8];
    }
    const float inv0 = (L0 > 0.f) ? kv_scale / L0 : 0.f;
    const float inv1 = (L1 > 0.f) ? kv_scale / L1 : 0.f;
    if (w.slot < 0) {
      __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + (int64_t)w.q_row * kHeads * kVDim;
      if constexpr (MODE == MLA_MODE_BF16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d = 64 * warp + 8 * i + 2 * c;
          *reinterpret_cast<uint32_t*>(ob + g * kVDim + d) = ptx::pack_bf16x2(o[i][0] * inv0, o[i][1] * inv0);
          *reinterpret_cast<uint32_t*>(ob + (g + 8) * kVDim + d) = ptx::pack_bf16x2(o[i][2] * inv1, o[i][3] * inv1);
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int d = 64 * warp + 32 * blk + 8 * c;  // this thread holds dims d .. d+7
          uint4 v0, v1;
          v0.x = ptx::pack_bf16x2(o[4 * blk + 0][0] * inv0, o[4 * blk + 1][0] * inv0);
          v0.y = ptx::pack_bf16x2(o[4 * blk + 2][0] * inv0, o[4 * blk + 3][0] * inv0);
          v0.z = ptx::pack_bf16x2(o[4 * blk + 0][1] * inv0, o[4 * blk + 1][1] * inv0);
          v0.w = ptx::pack_bf16x2(o[4 * blk + 2][1] * inv0, o[4 * blk + 3][1] * inv0);
          v1.x = ptx::pack_bf16x2(o[4 * blk + 0][2] * inv1, o[4 * blk + 1][2] * inv1);
          v1.y = ptx::pack_bf16x2(o[4 * blk + 2][2] * inv1, o[4 * blk + 3][2] * inv1);
          v1.z = ptx::pack_bf16x2(o[4 * blk + 0][3] * inv1, o[4 * blk + 1][3] * inv1);
          v1.w = ptx::pack_bf16x2(o[4 * blk + 2][3] * inv1, o[4 * blk + 3][3] * inv1);
          *reinterpret_cast<uint4*>(ob + g * kVDim + d) = v0;
          *reinterpret_cast<uint4*>(ob + (g + 8) * kVDim + d) = v1;
        }
      }
    } else {
      float* po = p.part_o + (int64_t)w.slot * kHeads * kVDim;
      if constexpr (MODE == MLA_MODE_BF16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int d = 64 * warp + 8 * i + 2 * c;
          *reinterpret_cast<float2*>(po + g * kVDim + d) = make_float2(o[i][0] * inv0, o[i][1] * inv0);
          *reinterpret_cast<float2*>(po + (g + 8) * kVDim + d) = make_float2(o[i][2] * inv1, o[i][3] * inv1);
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
          const int d = 64 * warp + 32 * blk + 8 * c;
          float* r0p = po + g * kVDim + d;
          float* r1p = po + (g + 8) * kVDim + d;
          *reinterpret_cast<float4*>(r0p) = make_float4(o[4 * blk + 0][0] * inv0, o[4 * blk + 1][0] * inv0,
                                                        o[4 * blk + 2][0] * inv0, o[4 * blk + 3][0] * inv0);
          *reinterpret_cast<float4*>(r0p + 4) = make_float4(o[4 * blk + 0][1] * inv0, o[4 * blk + 1][1] * inv0,
                                                            o[4 * blk + 2][1] * inv0, o[4 * blk + 3][1] * inv0);
          *reinterpret_cast<float4*>(r1p) = make_float4(o[4 * blk + 0][2] * inv1, o[4 * blk + 1][2] * inv1,
                                                        o[4 * blk + 2][2] * inv1, o[4 * blk + 3][2] * inv1);
          *reinterpret_cast<float4*>(r1p + 4) = make_float4(o[4 * blk + 0][3] * inv1, o[4 * blk + 1][3] * inv1,
                                                            o[4 * blk + 2][3] * inv1, o[4 * blk + 3][3] * inv1);
        }
      }
      if (warp == 0 && c == 0) {
        float* pl = p.part_lse + (int64_t)w.slot * kHeads;
        pl[g] = (L0 > 0.f) ? m_run[0] + __log2f(L0) : -INFINITY;
        pl[g + 8] = (L1 > 0.f) ? m_run[1] + __log2f(L1) : -INFINITY;
      }
    }
  }

  if (timed_out) {
    if (tid == 0) record_error(p.err, MLA_ERR_TIMEOUT);
    // Let copies still in flight land before the CTA's shared memory goes away.
    const int issued = min(n_tiles, tile + C::kStages - 1);
    for (int k = tile; k < issued; ++k)
      (void)ptx::mbar_wait_bounded(bar0 + 8u * (k % C::kStages), (uint32_t)(k / C::kStages) & 1u, kDrainLimitNs);
  }
}

template <int MODE, bool kPaged>
int launch_stage1_tp(const DecodeArgs& a, const DevicePlan& p, const uint8_t* zero_row, cudaStream_t stream) {
  // the shared-memory opt-in is set once per device and instance (an idempotent
  // call: threads that race to it both make it, and the flags are atomic)
  static std::atomic<bool> configured[64] = {};
  const int smem_bytes = Smem<MODE>::kBytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(mla_stage1_kernel<MODE, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return (int)e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.num_ctas <= 0) return 0;
  // programmatic stream serialisation: the prologue may overlap the previous kernel's tail
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, mla_stage1_kernel<MODE, kPaged>, a, p, zero_row);
}

template <int MODE>
int launch_stage1_t(const DecodeArgs& a, const DevicePlan& p, const uint8_t* zero_row, cudaStream_t stream) {
  return a.page_size > 1 ? launch_stage1_tp<MODE, true>(a, p, zero_row, stream)
                         : launch_stage1_tp<MODE, false>(a, p, zero_row, stream);
}

}  // namespace

int launch_stage1(int dtype_mode, const DecodeArgs& a, const DevicePlan& p, const void* zero_row, void* stream) {
  const uint8_t* z = static_cast<const uint8_t*>(zero_row);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype_mode == MLA_MODE_BF16) return launch_stage1_t<MLA_MODE_BF16>(a, p, z, s);
  // fp8 and a16w8 run on the tensor-memory kernel unless the plan asks for the warp-level one
  if (dtype_mode == MLA_MODE_A16W8)
    return p.fp8_kernel == 1 ? launch_stage1_t<MLA_MODE_A16W8>(a, p, z, s) : launch_stage1_a16w8_umma(a, p, stream);
  if (p.fp8_kernel == 1) return launch_stage1_t<MLA_MODE_FP8>(a, p, z, s);
  return launch_stage1_fp8_umma(a, p, stream);
}

}  // namespace mla
