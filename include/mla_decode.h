/*
 * mla_decode.h — C ABI of the GB300 (sm_103a) MLA decode library
 * (libmla_decode.so).
 *
 * The operation (kernelbot amd-mixed-mla submission 689529 "MLA decode V3",
 * module constants and custom_kernel): single-token decode of DeepSeek-style
 * Multi-head Latent Attention. 16 query heads share one KV head; a KV row is
 * 576 values (512-wide latent + 64-wide rope part); for sequence b and head h
 *   s_t      = sm_scale * <q[b,h,:], kv[row_t,:]>            (all 576 dims)
 *   out[b,h] = sum_t softmax_t(s) * kv[row_t, 0:512]          (first 512 dims)
 * with row_t = kv_indices[kv_indptr[b] + t] for 0 <= t < kv_indptr[b+1] -
 * kv_indptr[b] (page_size = 1: every page is one row; mla_decode_paged takes
 * pages of several rows). The pages' V6c and
 * v86 submissions run it as a persistent stage-1 kernel over a precomputed
 * work list followed by a split reduce (submission 690201 "V6c",
 * custom_kernel: direct stage1 and reduce calls; _build_cache: metadata and
 * cached partial buffers); this library keeps that split: a host planner
 * (mla_decode_plan) and a device pass (mla_decode = stage 1 + reduce).
 *
 * Conventions for every entry point:
 *  - Return value: MLA_OK (0) or a negative mla_status. No C++ exception
 *    crosses this boundary. mla_strerror() names a status.
 *  - "device" pointers are CUDA global memory of the current device, owned
 *    by the caller unless stated; "host" pointers are ordinary host memory.
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Device work is asynchronous on that stream; nothing here synchronises
 *    the stream except mla_plan_check_error().
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Problem constants fixed by the pages (V3 module constants). */
#define MLA_NUM_HEADS 16
#define MLA_NUM_KV_HEADS 1
#define MLA_QK_HEAD_DIM 576
#define MLA_V_HEAD_DIM 512
#define MLA_PAGE_SIZE 1 /* the row-addressed layout of mla_decode; mla_decode_paged takes any page size */

/* Value modes (dtype_mode argument). */
enum mla_dtype_mode {
  /* q bf16 [B,16,576], kv bf16 [slots,576]; kv_scale ignored. The pages'
     non-persistent bf16 path (submission 641982 "v86", custom_kernel). */
  MLA_MODE_BF16 = 0,
  /* q bf16 [B,16,576] is cast inside the kernel to OCP fp8 e4m3fn with scale 1
     (round to nearest even; magnitudes above 448 saturate) — the direct cast of
     V3 / V6c custom_kernel; kv holds e4m3fn bytes [slots,576] with one fp32
     per-tensor dequantisation scale *kv_scale (kv_data["fp8"] = (buffer,
     scale)). Scores use q8 . k8 * sm_scale * kv_scale; out is scaled by
     kv_scale. */
  MLA_MODE_FP8 = 1,
  /* "a16w8" (submission 598454 "v12", docstring: activations in their original
     precision, KV in fp8): q bf16 [B,16,576] used at bf16 precision (converted
     to f16 inside the kernel: exact for 2^-14 <= |q| < 65520, saturating at
     65504 beyond), kv e4m3fn bytes [slots,576] with *kv_scale as in
     MLA_MODE_FP8. Runs on the warp-level kernel (the 5th-generation tensor
     cores take no bf16 x e4m3 product). */
  MLA_MODE_A16W8 = 2
};

/* Status codes. */
enum mla_status {
  MLA_OK = 0,
  MLA_ERR_ARG = -1,           /* null pointer, negative size, bad batch or num_sms */
  MLA_ERR_DTYPE = -2,         /* unknown dtype_mode */
  MLA_ERR_PLAN_MISMATCH = -3, /* device kv_indptr disagrees with the plan (reported by the kernel) */
  MLA_ERR_CUDA = -4,          /* a CUDA runtime call failed */
  MLA_ERR_TIMEOUT = -5,       /* a bounded wait inside a kernel gave up (kernel returned early) */
  MLA_ERR_ALIGN = -6,         /* q, kv or out not 16-byte aligned */
  MLA_ERR_NOMEM = -7,         /* device or host allocation failed while planning */
  MLA_ERR_INDEX = -8,         /* a kv_indices entry lies outside [0, num_kv_slots) (reported by the kernel) */
  MLA_ERR_DEVICE = -9,        /* no usable sm_103 device, or the plan belongs to another device */
  MLA_ERR_INDPTR = -10,       /* host kv_indptr not non-decreasing from 0, or a sequence too long */
  MLA_ERR_NOALLOC_LIMIT = -11 /* mla_decode_noalloc: the request needs more than its fixed scratch holds */
};

/* Opaque plan: split-KV work list, reduce map and the partial-result
   workspace for one (batch, kv_indptr, num_sms) shape. Owned by the library. */
typedef struct mla_plan mla_plan;

/* Planner tunables (mla_decode_plan_ex). Zero in a field selects its default. */
typedef struct mla_plan_options {
  int64_t num_kv_slots;   /* rows in the KV pool; kv_indices are checked against it in the
                             kernel (out-of-range rows are skipped and MLA_ERR_INDEX recorded).
                             0 = unchecked (the plain mla_decode_plan) */
  int min_rows_per_split; /* smallest KV chunk the planner cuts (default 64) */
  int granularity;        /* work is balanced in units of this many rows, and chunk boundaries fall on
                             multiples of it from the sequence start (default 64: the warp-level kernels'
                             tile, half the tensor-memory kernel's) */
  int ctas_per_sm;        /* persistent CTAs per SM (default 1) */
  int fp8_kernel;         /* fp8 stage-1 kernel: 0 = 5th-generation tensor cores (tcgen05 + TMA, default),
                             1 = warp-level mma.sync (kept for comparison) */
  int fp8_issuers;        /* tcgen05 kernel's MMA issue: 2 = two issuing threads (scores, P.V) and two
                             loader warps (default, faster on every layout measured); 1 = one issuing
                             thread and three loader warps, kept for comparison. 0 = default. Results
                             are identical either way. */
  int item_cost_rows;     /* balancing: each work item a CTA starts (a sequence piece, per query token)
                             counts as this many extra KV rows when the planner evens out the CTAs'
                             work (an item boundary costs an epilogue and a pipeline refill). 0 = default
                             (256, about two tiles' time measured on fp8 B=64 L=8192); negative = none,
                             which divides the rows alone evenly. */
  int token_parallel;     /* several query tokens (mla_decode_plan_multi): when every sequence with KV rows
                             has the same number Q > 1 of query tokens, plan the row ranges for one
                             token and give each range Q CTAs, one per token, which read the same rows
                             at the same time (from HBM once, from L2 for the others). 0 = default (on);
                             negative = off: each range's tokens run back to back in one CTA. */
  int token_pairs;        /* several query tokens (mla_decode_plan_multi): when every sequence with KV rows
                             has the same even number Q of query tokens, the plan also holds a work list
                             in token pairs: tokens 2v and 2v+1 of a sequence in one pass over their
                             rows (both queries in one 32-column score MMA), which reads each KV tile
                             once for two tokens; token_parallel then applies to the Q/2 pairs.
                             mla_decode_multi uses it for MLA_MODE_FP8 on the tensor-core kernel
                             (fp8_kernel 0), and the ordinary list for every other decode. 0 = default
                             (on); negative = off; positive = on. */
} mla_plan_options;

/* Read-only description of a plan. */
typedef struct mla_plan_info {
  int batch;
  int num_ctas;           /* stage-1 grid size (persistent CTAs that received work) */
  int num_work_items;     /* (sequence, KV chunk) items in the work list */
  int num_partial_slots;  /* partial (O, LSE) slots in the workspace */
  int num_split_seqs;     /* sequences whose chunks are merged by the reduce kernel */
  int device;             /* CUDA device the plan's buffers live on */
  int64_t total_rows;     /* sum of the sequence lengths */
  int64_t max_rows_per_cta;
  size_t workspace_bytes; /* device bytes the plan owns */
  int token_pairs;        /* 1: the plan also holds a token-pair work list (the other fields describe the
                             ordinary list) */
} mla_plan_info;

/*
 * mla_decode_plan — host split-KV planner (the persistent-mode metadata of the
 * pages: get_mla_metadata_info_v1 / get_mla_metadata_v1 in submission 598454
 * "v12", _get_or_compute_metadata, and the cached logits / attn_lse buffers of
 * 690201 "V6c", _build_cache).
 *   batch          number of sequences B (>= 0).
 *   kv_indptr_host host int32 [B+1]: kv_indptr[0] = 0, non-decreasing; sequence b
 *                  owns kv_indices[kv_indptr[b] .. kv_indptr[b+1]). Read only
 *                  during the call.
 *   num_sms        SMs to spread the work over (<= 0: query the current device).
 *   plan_out       receives the plan. Plans are cached by (device, batch,
 *                  kv_indptr contents, num_sms, options): an identical request
 *                  returns the same plan with its reference count raised.
 * Allocates device memory (work list, reduce map, fp32 partial O [slots,16,512]
 * and LSE [slots,16], an error word) on the current device; synchronises the
 * device once to upload the work list. Errors: MLA_ERR_ARG, MLA_ERR_INDPTR,
 * MLA_ERR_NOMEM, MLA_ERR_CUDA, MLA_ERR_DEVICE.
 */
int mla_decode_plan(int batch, const int32_t* kv_indptr_host, int num_sms, mla_plan** plan_out);

/* mla_decode_plan with tunables (options may be NULL = defaults). */
int mla_decode_plan_ex(int batch, const int32_t* kv_indptr_host, int num_sms, const mla_plan_options* options,
                       mla_plan** plan_out);

/* Drop one reference to a plan; the last reference frees its device memory.
   The caller must ensure no decode using the plan is still in flight. */
int mla_plan_release(mla_plan* plan);

/* Fill *info with the plan's shape. */
int mla_plan_get_info(const mla_plan* plan, mla_plan_info* info);

/* The same release under the name the split-KV workspace is often given a
   destroy call by: drops one reference; the last one frees the plan's device
   memory. Returns MLA_OK or MLA_ERR_ARG (NULL or unknown plan). */
int mla_plan_destroy(mla_plan* plan);

/* Device bytes the plan owns (work list, reduce map, fp32 partials, error
   word; mla_plan_info.workspace_bytes). 0 for a NULL plan. */
size_t mla_plan_workspace_bytes(const mla_plan* plan);

/*
 * mla_decode — one decode call: stage 1 (+ reduce when any sequence is split).
 *   q          device bf16 [B,16,576], row-major, 16-byte aligned.
 *   kv         device [num_slots,576] row-major: bf16 (MLA_MODE_BF16) or e4m3fn
 *              bytes (MLA_MODE_FP8, MLA_MODE_A16W8); 16-byte aligned.
 *   kv_scale   device fp32 [1]: fp8 dequantisation scale (ignored in bf16 mode,
 *              may then be NULL).
 *   kv_indptr  device int32 [B+1], equal to the host array the plan was built
 *              from (the kernel checks each sequence length it touches and
 *              records MLA_ERR_PLAN_MISMATCH, skipping that work, if not).
 *   kv_indices device int32 [kv_indptr[B]]: KV row of every token.
 *   out        device bf16 [B,16,512], 16-byte aligned; fully written (an empty
 *              sequence yields zeros).
 *   sm_scale   softmax scale (the pages use 1/sqrt(576)).
 *   dtype_mode an mla_dtype_mode.
 *   workspace  the plan from mla_decode_plan for this batch / kv_indptr.
 *   stream     cudaStream_t.
 * Never allocates, never synchronises. A plan's workspace serves one decode at
 * a time: decodes sharing a plan must be ordered (same stream or events).
 * Errors detected on the host return immediately (MLA_ERR_ARG, MLA_ERR_DTYPE,
 * MLA_ERR_ALIGN, MLA_ERR_DEVICE, MLA_ERR_CUDA for a failed launch); errors found
 * by the kernel are recorded in the plan's error word (mla_plan_check_error).
 */
int mla_decode(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
               const int32_t* kv_indices, void* out, float sm_scale, int dtype_mode, mla_plan* workspace,
               void* stream);

/*
 * mla_decode_stage1 — only the persistent stage-1 kernel of mla_decode (the
 * pages' direct mla_decode_stage1_asm_fwd call, submission 690201 "V6c",
 * custom_kernel). Sequences the plan keeps whole get their final bf16 output
 * in out; split sequences get fp32 partial (O, LSE) in the workspace, which
 * mla_decode_reduce then merges. Arguments as for mla_decode.
 */
int mla_decode_stage1(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
                      const int32_t* kv_indices, void* out, float sm_scale, int dtype_mode, mla_plan* workspace,
                      void* stream);

/*
 * mla_decode_reduce — LSE-combine of the split sequences' partial results into
 * bf16 out (the pages' mla_reduce_v1 call, submission 690201 "V6c",
 * custom_kernel): per head, L = log sum_s e^{lse_s} and
 * out = sum_s e^{lse_s - L} * O_s. No-op when the plan splits no sequence.
 */
int mla_decode_reduce(void* out, mla_plan* workspace, void* stream);

/*
 * mla_plan_check_error — synchronise stream, read and clear the error word the
 * kernels set (MLA_OK, MLA_ERR_TIMEOUT, MLA_ERR_PLAN_MISMATCH, MLA_ERR_INDEX).
 */
int mla_plan_check_error(mla_plan* plan, void* stream);

/*
 * mla_plan_compute_host — the planner alone, on the host, with no CUDA call
 * (for inspection and testing; mla_decode_plan runs the same code).
 *   counts      host int32 [4] (required): number of work items, CTAs that get
 *               work, partial slots, split sequences.
 *   items       host int32 [items_cap][5] or NULL: per work item (sequence b,
 *               first row, end row, partial slot or -1 for a final write,
 *               sequence length), grouped by CTA in CTA order.
 *   work_indptr host int32 [indptr_cap] or NULL: CTA c owns items
 *               [work_indptr[c], work_indptr[c+1]); needs num_ctas + 1 entries.
 *   reduce      host int32 [reduce_cap][3] or NULL: per split sequence (b,
 *               first slot, slot count).
 * An array whose capacity is too small is left untouched (call once with NULL
 * arrays to size them). Errors: MLA_ERR_ARG, MLA_ERR_INDPTR, MLA_ERR_NOMEM.
 */
int mla_plan_compute_host(int batch, const int32_t* kv_indptr_host, int num_sms, const mla_plan_options* options,
                          int32_t* counts, int32_t* items, int items_cap, int32_t* work_indptr, int indptr_cap,
                          int32_t* reduce, int reduce_cap);

/*
 * mla_decode_noalloc — the same decode as mla_decode, for callers that cannot
 * allocate device memory. None of the cited submissions has such an entry point.
 *
 * Who needs it: code that is handed a stream and its buffers but may not call
 * cudaMalloc — for example a plug-in inside a framework whose caching
 * allocator has already reserved the device's memory, or a latency-critical
 * serving loop that cannot accept cudaMalloc's implicit device
 * synchronisation. Such a caller cannot build an mla_plan (mla_decode_plan
 * allocates the plan's workspace). This call instead plans on the host into
 * stack arrays and keeps the work list and the fp32 partial results in one
 * fixed array of device memory inside the library: 16 MiB, present on every
 * GPU that loads the library until the process exits. It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Limits: batch <= 1024 sequences and at most 500 partial results of split
 * sequences per call (the split targets one chunk per SM, so a split sequence
 * usually needs two or three). Larger requests return MLA_ERR_NOALLOC_LIMIT
 * before any device work is queued.
 *
 * Arguments as for mla_decode, plus:
 *   kv_indptr_host host int32 [batch+1]: the same offsets as the device kv_indptr
 *                  (the split is planned from it on every call).
 *   batch          number of sequences.
 *   num_kv_slots   rows in the KV pool; kv_indices are checked against it in the
 *                  kernel (0 = unchecked).
 *   status_dev     device int owned by the caller. This call sets it to 0 on the
 *                  stream; the kernels then record the first error they detect
 *                  (MLA_ERR_TIMEOUT, MLA_ERR_PLAN_MISMATCH, MLA_ERR_INDEX).
 * The first call on a device does a one-time set-up: it resolves the array's
 * device address and clears part of it, and synchronises the device. Make that
 * first call before any stream capture; while `stream` is being captured the
 * set-up is not attempted (MLA_ERR_CUDA), and a set-up that failed is retried
 * by the next call. Every call reuses the same array, which keeps the last
 * call's contents: calls whose device work overlaps (on different streams, or
 * unordered) race on it and corrupt each other's results.
 * Host costs: each call plans into about 93 KB of the calling thread's stack
 * (give threads with small stacks room for it), and uploads the work list
 * (up to about 90 KB) with cudaMemcpyAsync from that pageable memory, which the
 * runtime stages before returning and which can make the call wait for work
 * queued earlier on the stream.
 * Errors returned directly: MLA_ERR_ARG, MLA_ERR_DTYPE, MLA_ERR_ALIGN,
 * MLA_ERR_INDPTR, MLA_ERR_DEVICE, MLA_ERR_CUDA, MLA_ERR_NOALLOC_LIMIT.
 */
int mla_decode_noalloc(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr_host,
                       const int32_t* kv_indptr, const int32_t* kv_indices, int batch, int64_t num_kv_slots,
                       void* out, float sm_scale, int dtype_mode, int* status_dev, void* stream);

/*
 * Paged KV layout (kernelbot amd-mixed-mla submission 641982 "v86",
 * _run_a8w8, and 598454 "v12", custom_kernel: the KV buffer viewed as
 * [num_pages, page_size, 1, 576], kv_indptr // page_size, page ids in
 * kv_indices, kv_last_page_lens). Sequence b owns pages
 * kv_indices[kv_indptr[b] .. kv_indptr[b+1]); its last page holds
 * kv_last_page_len[b] tokens (1 <= len <= page_size), every other page holds
 * page_size. Token t is row kv_indices[kv_indptr[b] + t / page_size] *
 * page_size + t % page_size of the buffer. The rows of a last page past its
 * length never reach the result (they may hold anything, NaN codes included),
 * but the fp8 tensor-core kernel may load them: with pages of 16, 32 or 64
 * rows it loads whole pages, so every listed page must lie whole inside the
 * buffer.
 *
 * mla_decode_plan_paged — the planner for that layout.
 *   kv_indptr_host        host int32 [B+1] page offsets (0 first, non-decreasing).
 *   kv_last_page_len_host host int32 [B] (may be NULL when page_size is 1).
 *   page_size             tokens per page (>= 1).
 *   options->num_kv_slots counts ROWS of the buffer (num_pages * page_size).
 * Plans are cached by layout as well; a paged plan serves only
 * mla_decode_paged with the same page_size (any other decode call returns
 * MLA_ERR_ARG). Errors as mla_decode_plan, plus MLA_ERR_INDPTR for a last page
 * length outside [1, page_size] or a sequence longer than 2^31 - 1 tokens.
 */
int mla_decode_plan_paged(int batch, const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                          int page_size, int num_sms, const mla_plan_options* options, mla_plan** plan_out);
/*
 * mla_decode_paged — mla_decode over the paged layout.
 *   kv               device [num_pages * page_size, 576] (bf16 or e4m3 bytes).
 *   kv_indptr        device int32 [B+1] page offsets, equal to the plan's.
 *   kv_indices       device int32 page ids.
 *   kv_last_page_len device int32 [B], equal to the plan's (may be NULL when
 *                    page_size is 1). The kernel recomputes every token count it
 *                    touches and records MLA_ERR_PLAN_MISMATCH, skipping that work,
 *                    when it differs from the plan's.
 *   page_size        must equal the plan's.
 * Other arguments, ownership, ordering and errors as for mla_decode. A page id
 * whose rows fall outside [0, num_kv_slots) (when the plan was given the pool
 * size) is read as zeros and recorded as MLA_ERR_INDEX.
 */
int mla_decode_paged(const void* q, const void* kv, const float* kv_scale, const int32_t* kv_indptr,
                     const int32_t* kv_indices, const int32_t* kv_last_page_len, int page_size, void* out,
                     float sm_scale, int dtype_mode, mla_plan* workspace, void* stream);
/* mla_plan_compute_host for the paged layout (same outputs; token offsets in items). */
int mla_plan_compute_host_paged(int batch, const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                                int page_size, int num_sms, const mla_plan_options* options, int32_t* counts,
                                int32_t* items, int items_cap, int32_t* work_indptr, int indptr_cap,
                                int32_t* reduce, int reduce_cap);
/*
 * Several query tokens per sequence (the pages' qo_indptr / max_seqlen_q:
 * submission 690201 "V6c", _build_cache builds qo_indptr = arange(B+1) *
 * q_seq_len for the stage-1 call; is_causal is set in 689529 "V3",
 * _get_or_build_cache). Sequence b has q_b = qo_indptr[b+1] - qo_indptr[b]
 * query tokens, rows qo_indptr[b] .. qo_indptr[b+1]-1 of q [qo_indptr[B],16,576]
 * and out [qo_indptr[B],16,512]. They are the sequence's last q_b tokens: with
 * causal != 0, query token j attends to the first max(0, L_b - q_b + j + 1) of
 * the sequence's L_b KV tokens (the lower-right-aligned causal mask), else to
 * all of them. A query token that sees no KV token gets zeros. KV addressing is
 * the paged layout above; page_size 1 with kv_last_page_len NULL is plain row
 * addressing.
 *
 * When every sequence with KV rows has the same number Q > 1 of query tokens
 * (the usual speculative-decoding batch), the planner cuts the rows into
 * ranges for one token and gives each range Q CTAs, one per token, side by
 * side: they read each row at about the same time, from HBM once and from L2
 * for the other tokens (option token_parallel). Otherwise one CTA processes the
 * query tokens of a range back to back on the same rows, which find them in L2
 * only while the CTAs' ranges fit in it. When that number Q is even, the plan
 * also holds a work list in token pairs, which fp8 decodes on the tensor-core
 * kernel use: two tokens per pass over their rows (option token_pairs).
 *
 * mla_decode_plan_multi — the planner for that layout (host arrays as for
 *   mla_decode_plan_paged, plus qo_indptr_host [B+1], 0 first, non-decreasing).
 *   A multi-token plan serves only mla_decode_multi with the same page_size.
 *   Errors as mla_decode_plan_paged, MLA_ERR_INDPTR also for a bad qo_indptr.
 */
int mla_decode_plan_multi(int batch, const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                          const int32_t* kv_last_page_len_host, int page_size, int causal, int num_sms,
                          const mla_plan_options* options, mla_plan** plan_out);
/*
 * mla_decode_multi — decode of every query token.
 *   q          device bf16 [qo_indptr[B], 16, 576]; out device bf16 [qo_indptr[B], 16, 512].
 *   qo_indptr  device int32 [B+1], equal to the plan's (the kernel checks each
 *              item's query row against it and records MLA_ERR_PLAN_MISMATCH,
 *              skipping that work, if not).
 *   Other arguments, ownership, ordering and errors as mla_decode_paged.
 */
int mla_decode_multi(const void* q, const void* kv, const float* kv_scale, const int32_t* qo_indptr,
                     const int32_t* kv_indptr, const int32_t* kv_indices, const int32_t* kv_last_page_len,
                     int page_size, void* out, float sm_scale, int dtype_mode, mla_plan* workspace, void* stream);
/* mla_plan_compute_host for multi-token plans: items as int32 [items_cap][8] =
   (sequence, first token, end token, partial slot or -1, sequence length,
   query row, query token within the sequence, pair field), and the reduce map
   as int32 [reduce_cap][4] = (query row, first slot, slots, slot stride).
   The pair field is 0 in ordinary plans. In token-pair plans an item with pair
   field >= 0 covers query rows r and r + 1 (tokens j and j + 1): row r sees
   tokens [first, pair field), row r + 1 tokens [first, end), and their partial
   slots are slot and slot + 1; -1 marks an item of one query row (a sequence
   without KV rows). The slot stride is 0 (consecutive slots) or 2 (a row of a
   token pair). */
int mla_plan_compute_host_multi(int batch, const int32_t* qo_indptr_host, const int32_t* kv_indptr_host,
                                const int32_t* kv_last_page_len_host, int page_size, int causal, int num_sms,
                                const mla_plan_options* options, int32_t* counts, int32_t* items, int items_cap,
                                int32_t* work_indptr, int indptr_cap, int32_t* reduce, int reduce_cap);
/* Human-readable name of a status code (static string). */
const char* mla_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
