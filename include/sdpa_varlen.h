/*
 * sdpa_varlen.h - C interface of the GB300 (sm_103a) length-aware GQA attention library.
 *
 * The operation ("[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV
 * columns", PR description, with the #24073 and #24074 commit messages of its stack):
 * each resident sequence owns one column of a K store and a V store laid out
 * [rows, cols, Hkv, D]; a device segment table seq_info Int32[S, 4] =
 * (q_start, q_len, col, kv_end) maps packed query rows [q_start, q_start + q_len) to
 * column `col` holding `kv_end` positions.  Query row i of a segment sits at position
 * p = kv_end - q_len + i (the step's queries are its last q_len positions, written into
 * the store before attention reads it).  Position j of a column lives in store row
 * j % rows (ring layers have fewer rows than positions).  A query sees key j when
 * j < kv_end, and j <= p if causal, and j > p - window if window > 0.  Query head h reads
 * KV head h / (Hq / Hkv).  out[t, h, :] = sum_j softmax_j(scale * q . k_j) v_j.
 * Rows no valid segment covers are written as 0, and so are rows that see no key
 * ("[CUDA] Use Triton TMA for long-context causal prefill", Summary: fully masked rows
 * keep finite outputs).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library keeps no
 *    reference to them after the call returns and allocates no device memory.
 *  - bf16 tensors hold IEEE bfloat16 values (uint16 bit patterns).
 *  - Strides are in elements.  The innermost (head-dim) stride is always 1.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream).  No call
 *    but the status read-back sdpa_workspace_status synchronises the host, so all the others
 *    may be captured into a CUDA graph.  Lengths are read on the device: one captured graph
 *    serves any seq_info contents.
 *  - The return value reports argument checks (made before any CUDA call) and launch
 *    errors.  Errors inside a segment table are reported through `status_dev`.
 *  - sdpa_last_error() returns a thread-local message describing the last failure.
 */
#ifndef SDPA_VARLEN_H
#define SDPA_VARLEN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side return codes. */
typedef enum sdpa_status {
  SDPA_OK = 0,
  SDPA_ERR_NULL = 1,      /* a required pointer is NULL                              */
  SDPA_ERR_SHAPE = 2,     /* a size is out of range (T, S, rows, cols, heads < 0 ...) */
  SDPA_ERR_HEAD_DIM = 3,  /* D is not 64, 128 or 256                                 */
  SDPA_ERR_GQA = 4,       /* Hq is not a multiple of Hkv, or Hq / Hkv > 128          */
  SDPA_ERR_STRIDE = 5,    /* a row/head stride is not a multiple of 8 elements       */
  SDPA_ERR_ALIGN = 6,     /* a tensor pointer is not 16-byte aligned                 */
  SDPA_ERR_WORKSPACE = 7, /* workspace NULL or smaller than the query says           */
  SDPA_ERR_ARG = 8,       /* window < 0, scale not finite, unknown route policy      */
  SDPA_ERR_CUDA = 9       /* a CUDA call failed; see sdpa_last_error()               */
} sdpa_status;

/* Device status bits, ORed into *status_dev by sdpa_varlen.  A segment with any of the
 * first four bits is skipped and its rows are written as 0. */
#define SDPA_SEG_BAD_QRANGE 1 /* q_len < 0, q_start < 0 or q_start + q_len > T            */
#define SDPA_SEG_BAD_COL 2    /* col outside [0, cols)                                    */
#define SDPA_SEG_BAD_KV 4     /* kv_end < 0                                               */
#define SDPA_SEG_SPAN 8       /* the keys the segment's rows see span more than `rows`
                                 store rows, so a ring has already overwritten one of them:
                                 span = window > 0 ? min(kv_end, q_len + window - 1) : kv_end */
#define SDPA_SEG_OVERLAP 16   /* two valid segments share a packed row: every row of both
                                 has an unspecified output                                */
#define SDPA_DEV_TIMEOUT 32   /* a bounded device wait gave up; the output is unspecified */

/* Route policy (process-wide).  AUTO sends segments with q_len * (Hq / Hkv) >= 128 to the
 * tensor-memory prefill kernel when the call's such segments hold at least 2^30 of work
 * (sum of packed rows * needed key span, times Hkv * D: below it that kernel's fixed cost
 * outweighs its speed), and everything else to the split-K kernel; the other two force
 * every segment onto one kernel (used to compare the kernels against each other). */
#define SDPA_ROUTE_AUTO 0
#define SDPA_ROUTE_SPLITK 1
#define SDPA_ROUTE_PREFILL 2

/* Bytes of device workspace sdpa_varlen needs for these bounds.  Depends only on sizes
 * the host knows (never on seq_info contents), so a graph can be captured once. */
size_t sdpa_varlen_workspace_bytes(int64_t T, int Hq, int Hkv, int D, int S);

/*
 * Length-aware GQA attention over a per-sequence KV column store.
 *
 *  q          [T, Hq, D] bf16; element (t, h, d) at q[t*q_row_stride + h*q_head_stride + d].
 *  k_store,   [rows, cols, Hkv, D] bf16, contiguous: element (r, c, h, d) at
 *  v_store    ((r*cols + c)*Hkv + h)*D + d.
 *  seq_info   [S, 4] int32, contiguous, device memory: (q_start, q_len, col, kv_end).
 *  causal     nonzero: key j must satisfy j <= p.
 *  window     0: no window; > 0: key j must satisfy j > p - window.
 *  scale      multiplies q . k before the softmax (for example 1/sqrt(D)).
 *  out        [T, Hq, D] bf16 with its own strides; every row t in [0, T) is written.
 *  workspace  device scratch of at least sdpa_varlen_workspace_bytes(T, Hq, Hkv, D, S)
 *             bytes, 256-byte aligned; its contents need no initialisation and are
 *             overwritten.  Two calls that run at the same time need two workspaces.
 *  status_dev NULL, or a device int32 the call ORs SDPA_SEG_* / SDPA_DEV_* bits into
 *             (it is never cleared by the library).
 *  stream     cudaStream_t to enqueue on.
 *
 * Requirements: D in {64, 128, 256}; Hq % Hkv == 0 and Hq / Hkv <= 128; T, S >= 0;
 * rows, cols >= 1; q, out, stores and workspace 16-byte aligned; row and head strides
 * multiples of 8 elements; window >= 0; scale finite.
 */
sdpa_status sdpa_varlen(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                        int64_t q_head_stride, const void* k_store, const void* v_store,
                        int64_t rows, int cols, int Hkv, const int32_t* seq_info, int S,
                        int causal, int window, float scale, void* out, int64_t o_row_stride,
                        int64_t o_head_stride, void* workspace, size_t ws_bytes,
                        int32_t* status_dev, void* stream);

/*
 * Write the step's keys and values, then attend: the in-graph slot write followed by the
 * attention of "[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV
 * columns" (#24074 commit message in its stack: slot (position % rows) * columns + col).
 *
 *  k_new, v_new    device bf16, [T, Hkv, D] packed like q: row t holds the new key / value
 *                  of packed query row t, every KV head; element (t, h, d) at
 *                  t*new_row_stride + h*new_head_stride + d; 16-byte aligned; strides
 *                  non-negative multiples of 8 elements; read only.
 *  k_store, v_store  as for sdpa_varlen, but written: for every live segment (valid and
 *                  not sharing a packed row with another valid segment), packed row
 *                  q_start + i, at position p = kv_end - q_len + i >= 0, is copied to store
 *                  row p % rows of column col, all KV heads.  Rows of invalid or
 *                  overlapping segments, uncovered rows and rows with p < 0 write nothing.
 *                  Two live segments that write the same (row, column) cell leave it
 *                  holding one of the two rows.
 * Every other argument, the attention that follows (it reads the written rows) and the
 * status bits are those of sdpa_varlen; the write runs on the device between its
 * scheduler and its attention kernels, in the same stream (so a captured graph holds both).
 * Errors as sdpa_varlen, plus SDPA_ERR_NULL / _ALIGN / _STRIDE for k_new and v_new.
 */
sdpa_status sdpa_varlen_append(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                               int64_t q_head_stride, const void* k_new, const void* v_new,
                               int64_t new_row_stride, int64_t new_head_stride, void* k_store,
                               void* v_store, int64_t rows, int cols, int Hkv, const int32_t* seq_info,
                               int S, int causal, int window, float scale, void* out,
                               int64_t o_row_stride, int64_t o_head_stride, void* workspace,
                               size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * Attention with a mask mode per segment, so that causal target segments and non-causal
 * draft blocks of one step share one launch (the #24074 manifest of "[executorch][cuda] Add a
 * length-aware Triton SDPA over per-sequence KV columns" carries `causal` per model, false for
 * DFlash drafts; here the choice moves into the segment table).
 *
 *  seg_mode  device int32 [S, 2], 16-byte aligned: row s = (causal, window) of segment s,
 *            with the meanings of sdpa_varlen's causal (non-zero: causal) and window (W > 0
 *            keys counting the query's own; <= 0: no window).  Read on the device, so one
 *            captured graph serves any mix; a segment's validity (needed span <= rows) uses
 *            its own window.
 * Every other argument and the result are those of sdpa_varlen, whose causal / window
 * arguments this call replaces.  Errors as sdpa_varlen, plus SDPA_ERR_NULL for seg_mode.
 */
sdpa_status sdpa_varlen_modes(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                              int64_t q_head_stride, const void* k_store, const void* v_store,
                              int64_t rows, int cols, int Hkv, const int32_t* seq_info,
                              const int32_t* seg_mode, int S, float scale, void* out,
                              int64_t o_row_stride, int64_t o_head_stride, void* workspace,
                              size_t ws_bytes, int32_t* status_dev, void* stream);

/*
 * seq_clone: column dst_col takes over the first n positions of column src_col ("[executorch]
 * [cuda] Add a length-aware Triton SDPA over per-sequence KV columns", #24073 commit message
 * in its stack: seq_clone, a device copy of the source prefix).  Position j lives in store
 * row j % rows, so positions [max(0, n - rows), n) are copied: store rows [0, min(n, rows))
 * of the source column, every KV head, K and V, to the same rows of the destination column.
 * Other rows of the destination keep their contents; src_col == dst_col or n == 0 does
 * nothing.  k_store, v_store: [rows, cols, Hkv, D] contiguous bf16 device stores, 16-byte
 * aligned.  Enqueued on `stream` (cudaStream_t), no host synchronisation.
 * Errors: SDPA_ERR_NULL, _ALIGN, _SHAPE (rows, cols, Hkv < 1 or n < 0), _HEAD_DIM, _ARG
 * (a column outside [0, cols)), _CUDA.
 */
sdpa_status sdpa_seq_clone(void* k_store, void* v_store, int64_t rows, int cols, int Hkv, int D,
                           int src_col, int dst_col, int64_t n, void* stream);

/*
 * Dense causal GQA prefill ("[CUDA] Use Triton TMA for long-context causal prefill",
 * Operator-level performance table: B = 1, global causal, queries being the last Lq of
 * Lkv positions).  q [Lq, Hq, D], k and v [Lkv, Hkv, D] contiguous bf16; out [Lq, Hq, D]
 * contiguous bf16.  A [Lkv, Hkv, D] tensor is a column store with one column, so this is
 * sdpa_varlen with the single segment (0, Lq, 0, Lkv), which is passed by value (no
 * device table).  Requires Lq <= Lkv.  Workspace as for sdpa_varlen with T = Lq, S = 1.
 */
sdpa_status sdpa_causal_prefill(const void* q, const void* k, const void* v, int64_t Lq,
                                int64_t Lkv, int Hq, int Hkv, int D, float scale, void* out,
                                void* workspace, size_t ws_bytes, void* stream);

/* Set the process-wide route policy (SDPA_ROUTE_*).  Returns SDPA_ERR_ARG if unknown. */
sdpa_status sdpa_set_route_policy(int policy);

/* Timing hook for this thread's next calls.  `events` holds 5 cudaEvent_t handles (or is
 * NULL to switch the hook off); each call then records them on its stream at the kernel
 * boundaries: [0] before the scheduler, [1] before the prefill kernel, [2] before the
 * split-K kernel, [3] before the combine pass, [4] after it.  The caller owns the events.
 * Returns SDPA_ERR_ARG if n != 5 while events is non-NULL. */
sdpa_status sdpa_set_timing_events(void* const* events, int n);

/* Bytes of the device array that sdpa_varlen_splitk_static uses as its scratch (32 MiB).
 * Every GPU that loads the library holds this array until the process exits. */
#define SDPA_STATIC_SCRATCH_BYTES (32u << 20)

/*
 * sdpa_varlen for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this entry point exists for callers such as a runtime with a fixed memory
 * plan, a plugin that may not call cudaMalloc, or a binding with no device allocator, which
 * cannot provide sdpa_varlen's workspace.)
 *
 * Arguments and results are those of sdpa_varlen without `workspace`/`ws_bytes`; every
 * segment runs on the split-K kernel.  The scratch is a file-scope device array of
 * SDPA_STATIC_SCRATCH_BYTES inside the library; nothing is allocated.  Sizes whose scratch
 * does not fit return SDPA_ERR_WORKSPACE (sdpa_last_error() says how much they need).
 * The first call on each device looks up the array's device address (with that device
 * current) and configures the kernels: make that first call before any stream capture.
 * The address is kept until the process exits, which assumes the device's primary context
 * lives as long: after cudaDeviceReset on a device, do not call this entry point there again.
 * All calls on a device share the one array and it keeps the last call's contents; nothing
 * in it needs to start at zero, but calls that overlap on the GPU (different streams, or
 * graphs replayed at the same time) race on it and must be serialised by the caller.
 */
sdpa_status sdpa_varlen_splitk_static(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                                      int64_t q_head_stride, const void* k_store, const void* v_store,
                                      int64_t rows, int cols, int Hkv, const int32_t* seq_info, int S,
                                      int causal, int window, float scale, void* out,
                                      int64_t o_row_stride, int64_t o_head_stride, int32_t* status_dev,
                                      void* stream);

/*
 * Whether the tensor-memory prefill kernel can run for head dim D on the current device:
 * 1 yes, 0 no (every call then takes the split-K kernel, with the same results), -1 on a
 * CUDA error or a head dim outside {64, 128, 256} (message in sdpa_last_error).  The answer
 * is fixed once per device, on first use.
 */
int sdpa_prefill_available(int D);

/*
 * Status of the last call that used `workspace` (sdpa_varlen, _append, _modes or
 * sdpa_causal_prefill), for callers that passed no status_dev: the OR of the SDPA_SEG_* bits
 * its scheduler found and SDPA_DEV_TIMEOUT when one of its bounded device waits gave up (its
 * output is then unspecified).  Waits for `stream` (cudaStream_t) to finish, then copies the
 * word to *status_host, so it synchronises the host and cannot be captured in a graph; a
 * caller that checks every replay of a graph passes status_dev instead.  Errors:
 * SDPA_ERR_NULL, _ALIGN (workspace not 256-byte aligned), _WORKSPACE (ws_bytes smaller than
 * the header), _CUDA.
 */
sdpa_status sdpa_workspace_status(const void* workspace, size_t ws_bytes, int32_t* status_host, void* stream);

/* Message describing the last failure on this thread ("" if none). */
const char* sdpa_last_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int sdpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_VARLEN_H */
