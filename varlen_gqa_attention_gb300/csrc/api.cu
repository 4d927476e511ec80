// api.cu - the C interface: argument checks, workspace layout, launches.
//
// Every check runs before any CUDA call, so a bad argument never touches the device.  The
// launches are asynchronous and allocation-free, so a call can be captured in a CUDA graph;
// the device scheduler reads the segment table when the graph replays.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace sdpa {

static thread_local char g_err[512] = "";
static thread_local cudaEvent_t g_ev[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
static thread_local bool g_ev_on = false;

// Records timing event i on `st`.  Under stream capture the record must become an event
// node of the graph (cudaEventRecordExternal) so that it fires on every replay.
static cudaError_t mark(int i, cudaStream_t st) {
  if (!g_ev_on) return cudaSuccess;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(g_ev[i], st, cudaEventRecordExternal)
                                             : cudaEventRecord(g_ev[i], st);
}
static std::atomic<int> g_policy{SDPA_ROUTE_AUTO};

static sdpa_status fail(sdpa_status code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

void set_last_error(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Per-device launch facts, measured once.
struct DevInfo {
  bool ready = false;
  int sms = 0;
  int splitk_per_sm[3] = {0, 0, 0};  // D = 64, 128, 256
  bool prefill_ok[3] = {false, false, false};
};
static std::mutex g_mu;
static DevInfo g_dev[64];

static int d_index(int D) { return D == 64 ? 0 : D == 128 ? 1 : 2; }

static sdpa_status device_info(DevInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(SDPA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& di = g_dev[dev];
  if (!di.ready) {
    e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
    e = cudaFuncSetAttribute(sched_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sched_smem_bytes());
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "scheduler smem attribute: %s", cudaGetErrorString(e));
    // every kernel of a call asks for the whole shared-memory carveout, so that the SMs keep
    // one L1 / shared split from kernel to kernel (the clone kernel runs alone and keeps the
    // default split, its L1 to itself)
    const void* others[3] = {sched_kernel_ptr(), sched_small_kernel_ptr(), append_kernel_ptr()};
    for (const void* f : others) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "carveout attribute: %s", cudaGetErrorString(e));
    }
    const int Ds[3] = {64, 128, 256};
    for (int k = 0; k < 3; ++k) {
      const void* f = splitk_kernel_ptr(Ds[k]);
      const int smem = splitk_smem_bytes(Ds[k]);
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "smem attribute: %s", cudaGetErrorString(e));
      // two split-K CTAs per SM need the whole shared-memory carveout
      e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "carveout attribute: %s", cudaGetErrorString(e));
      int nb = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, f, kSplitkThreads, smem);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "occupancy: %s", cudaGetErrorString(e));
      di.splitk_per_sm[k] = nb > 0 ? nb : 1;
      e = cudaFuncSetAttribute(combine_kernel_ptr(Ds[k]), cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "carveout attribute: %s", cudaGetErrorString(e));
      const void* pf = prefill_kernel_ptr(Ds[k]);
      e = cudaFuncSetAttribute(pf, cudaFuncAttributeMaxDynamicSharedMemorySize, prefill_smem_bytes(Ds[k]));
      if (e == cudaSuccess) e = cudaFuncSetAttribute(pf, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      di.prefill_ok[k] = e == cudaSuccess;
      if (e != cudaSuccess) cudaGetLastError();  // leave no sticky error; split-K covers it
    }
    di.ready = true;
  }
  *out = di;
  return SDPA_OK;
}

// cuTensorMapEncodeTiled, fetched from the driver once (no link against libcuda).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    else
      cudaGetLastError();
  });
  return fn;
}

// TMA descriptors of q [T, Hq, D] (box: 64 dims x group heads x 128/group rows, i.e. one
// 128-row tile of packed (row, head) pairs) and of the stores [rows, cols, Hkv, D] (box:
// 64 dims x 1 head x 1 column x `bn` rows), all with 128-byte swizzle.
static bool make_tensor_maps(const void* q, int64_t T, int Hq, int D, int64_t q_rs, int64_t q_hs,
                             const void* k, const void* v, int64_t rows, int cols, int Hkv, int group,
                             int bn, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || T <= 0 || q_hs <= 0 || q_rs <= 0) return false;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const cuuint64_t qdim[3] = {(cuuint64_t)D, (cuuint64_t)Hq, (cuuint64_t)T};
  const cuuint64_t qstr[2] = {(cuuint64_t)q_hs * 2, (cuuint64_t)q_rs * 2};
  const cuuint32_t qbox[3] = {64, (cuuint32_t)group, (cuuint32_t)(kPrefillRows / group)};
  if (enc(mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)q, qdim, qstr, qbox, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t kdim[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t kstr[3] = {(cuuint64_t)D * 2, (cuuint64_t)Hkv * D * 2, (cuuint64_t)cols * Hkv * D * 2};
  const cuuint32_t kbox[4] = {64, 1, 1, (cuuint32_t)bn};
  for (int w = 0; w < 2; ++w) {
    if (enc(w ? mv : mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)(w ? v : k), kdim, kstr, kbox, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

struct Grids {
  int64_t splitk, prefill;
};
static Grids grids_for(const DevInfo& di, int D) {
  Grids g;
  g.splitk = (int64_t)di.sms * di.splitk_per_sm[d_index(D)];
  g.prefill = di.sms;
  return g;
}

sdpa_status check_common(int64_t T, int Hq, int Hkv, int D, int S, int64_t rows, int cols, int window,
                         float scale) {
  if (T < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || rows <= 0 || cols <= 0)
    return fail(SDPA_ERR_SHAPE, "bad sizes: T=%lld S=%d Hq=%d Hkv=%d rows=%lld cols=%d",
                (long long)T, S, Hq, Hkv, (long long)rows, cols);
  if (T > INT32_MAX || rows > INT32_MAX || (int64_t)Hq * T > ((int64_t)1 << 40))
    return fail(SDPA_ERR_SHAPE, "T or rows beyond 2^31-1");
  if (D != 64 && D != 128 && D != 256) return fail(SDPA_ERR_HEAD_DIM, "head dim %d not in {64,128,256}", D);
  if (Hq % Hkv != 0 || Hq / Hkv > 128)
    return fail(SDPA_ERR_GQA, "Hq=%d is not a multiple of Hkv=%d (group <= 128)", Hq, Hkv);
  if (window < 0) return fail(SDPA_ERR_ARG, "window %d < 0", window);
  if (!std::isfinite(scale)) return fail(SDPA_ERR_ARG, "scale is not finite");
  return SDPA_OK;
}

sdpa_status check_tensors(const void* q, const void* k, const void* v, void* out, const int32_t* seq_info,
                          int S, int64_t q_rs, int64_t q_hs, int64_t o_rs, int64_t o_hs) {
  if (!q || !k || !v || !out || (!seq_info && S > 0)) return fail(SDPA_ERR_NULL, "a required pointer is NULL");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || (seq_info && !aligned16(seq_info)))
    return fail(SDPA_ERR_ALIGN, "tensor pointers must be 16-byte aligned");
  if (q_rs % 8 || q_hs % 8 || o_rs % 8 || o_hs % 8 || q_rs < 0 || q_hs < 0 || o_rs < 0 || o_hs < 0)
    return fail(SDPA_ERR_STRIDE, "row/head strides must be non-negative multiples of 8 elements");
  return SDPA_OK;
}

struct TensorMaps {
  CUtensorMap q, k, v;
};

// Launch with programmatic stream serialisation (the kernel waits in-kernel for its
// predecessor), except while the timing hook records events between the kernels: an event
// between two kernels would only serialise them again, and each kernel is then timed alone.
static cudaError_t launch_k(const void* f, unsigned grid, unsigned block, void** args, size_t smem,
                            cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  if (pdl && !g_ev_on) {
    cfg.attrs = at;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelExC(&cfg, f, args);
}

// Whether a call may route segments to the prefill kernel: not under the split-K policy, and
// (automatic routing) not when no segment can fill a 128-row tile (T * group < 128) or the
// call cannot hold kPrefillMinWork of prefill work: that is at most packed rows * Hkv * D *
// the longest needed key span, which is at most the store's rows (longer spans are invalid)
// and, with a call-wide window, T + window - 1.  The scheduler takes the result as
// prefill_ok, so it never routes work to a prefill kernel that is not launched.
static bool prefill_launch(const SchedArgs& sa, int64_t T) {
  if (sa.policy == SDPA_ROUTE_SPLITK) return false;
  if (sa.policy == SDPA_ROUTE_PREFILL) return true;
  const int64_t packed = T * sa.group;
  int64_t span_max = sa.rows;
  if (!sa.seg_mode && sa.window > 0) span_max = std::min<int64_t>(span_max, T + sa.window - 1);
  return packed >= kPrefillRows && (double)packed * sa.Hkv * sa.D * (double)span_max >= (double)kPrefillMinWork;
}

static sdpa_status launch_all(const SchedArgs& sa, const AttnArgs& aa, int D, const Grids& g,
                              const TensorMaps& tm, const AppendArgs* ap, cudaStream_t st) {
  cudaError_t e = mark(0, st);
  if (e == cudaSuccess) {
    e = launch_sched(sa, st);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "scheduler launch: %s", cudaGetErrorString(e));
  }
  if (e == cudaSuccess && ap && sa.S > 0) {
    // the step's new keys and values, between the scheduler (whose segment records say
    // which segments are live) and the attention kernels that read them
    void* args[] = {(void*)ap};
    const int64_t per_seg = (aa.T + sa.S - 1) / sa.S;
    const int64_t chunks = per_seg * ap->Hkv * (ap->D / 8);
    const unsigned gy = (unsigned)std::min<int64_t>(256, std::max<int64_t>(1, chunks / (4 * kAppendThreads)));
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)sa.S, gy);
    cfg.blockDim = dim3(kAppendThreads);
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    if (!g_ev_on) {
      cfg.attrs = at;
      cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelExC(&cfg, append_kernel_ptr(), args);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
  }
  if (e == cudaSuccess) e = mark(1, st);
  // The prefill kernel is launched when the call's schedule may use it (prefill_ok, see
  // prefill_launch).  Chained to the scheduler (programmatic dependent launch: its launch
  // overlaps the scheduler) when the average segment fills less than one tile, so that the
  // launch is most likely empty; launched after the scheduler otherwise (measured: the
  // chained launch saves ~6 us on a decode step whose prefill kernel has nothing to do, and
  // costs ~5 us on prefill steps of a few tiles per CTA).
  const int64_t packed = aa.T * aa.group;
  const bool pf_possible = sa.prefill_ok;
  if (e == cudaSuccess && pf_possible) {
    void* args[] = {(void*)&aa, (void*)&tm.q, (void*)&tm.k, (void*)&tm.v};
    const bool chained = packed < (int64_t)kPrefillRows * std::max(sa.S, 1);
    e = launch_k(prefill_kernel_ptr(D), (unsigned)g.prefill, prefill_block_threads(D), args,
                 prefill_smem_bytes(D), st, chained);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  }
  if (e == cudaSuccess) e = mark(2, st);
  if (e == cudaSuccess) {
    void* args[] = {(void*)&aa};
    e = launch_k(splitk_kernel_ptr(D), (unsigned)g.splitk, kSplitkThreads, args, splitk_smem_bytes(D), st, true);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "split-K launch: %s", cudaGetErrorString(e));
  }
  if (e == cudaSuccess) e = mark(3, st);
  if (e == cudaSuccess && aa.T > 0) {
    void* args[] = {(void*)&aa};
    const int64_t warps = aa.T * aa.Hq;
    const int64_t blocks = std::min<int64_t>((warps * 32 + 255) / 256, 8 * (int64_t)g.prefill);
    e = launch_k(combine_kernel_ptr(D), (unsigned)blocks, 256, args, 0, st, true);
    if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
  }
  if (e == cudaSuccess) e = mark(4, st);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "timing event: %s", cudaGetErrorString(e));
  return SDPA_OK;
}

static sdpa_status run(const void* q, int64_t T, int Hq, int D, int64_t q_rs, int64_t q_hs,
                       const void* k, const void* v, int64_t rows, int cols, int Hkv,
                       const int32_t* seq_info, int S, const int32_t* inl, int causal, int window,
                       float scale, void* out, int64_t o_rs, int64_t o_hs, void* ws, size_t ws_bytes,
                       int32_t* status_dev, void* stream, const AppendArgs* ap = nullptr,
                       const int32_t* seg_mode = nullptr) {
  g_err[0] = 0;
  sdpa_status st = check_common(T, Hq, Hkv, D, S, rows, cols, window, scale);
  if (st) return st;
  // the dense entry passes its one segment by value: no table pointer to check
  if ((st = check_tensors(q, k, v, out, seq_info, inl ? 0 : S, q_rs, q_hs, o_rs, o_hs))) return st;
  if (!ws) return fail(SDPA_ERR_WORKSPACE, "workspace is NULL");
  if ((uintptr_t)ws % 256) return fail(SDPA_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (seg_mode && !aligned16(seg_mode)) return fail(SDPA_ERR_ALIGN, "seg_mode must be 16-byte aligned");

  DevInfo di;
  if ((st = device_info(&di))) return st;
  const Grids g = grids_for(di, D);
  Workspace W;
  const size_t need = layout_workspace((char*)ws, T, Hq, Hkv, D, S, g.splitk, g.prefill, &W);
  if (ws_bytes < need)
    return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes, %zu needed", ws_bytes, need);

  SchedArgs sa{};
  sa.seq_info = seq_info;
  sa.seg_mode = S > 0 ? seg_mode : nullptr;
  sa.S = S;
  sa.use_inline = inl != nullptr;
  if (inl)
    for (int i = 0; i < 4; ++i) sa.inl[i] = inl[i];
  sa.T = T;
  sa.rows = rows;
  sa.cols = cols;
  sa.Hkv = Hkv;
  sa.group = Hq / Hkv;
  sa.causal = causal ? 1 : 0;
  sa.window = window;
  sa.D = D;
  sa.policy = g_policy.load();
  TensorMaps tm;
  const int group = Hq / Hkv;
  const bool group_fits = group <= kPrefillRows && (kPrefillRows % group) == 0;
  sa.tile_pf = prefill_tile_keys(D);
  sa.prefill_ok = di.prefill_ok[d_index(D)] && group_fits && prefill_launch(sa, T) &&
                  make_tensor_maps(q, T, Hq, D, q_rs, q_hs, k, v, rows, cols, Hkv, group, sa.tile_pf,
                                   &tm.q, &tm.k, &tm.v);
  sa.grid[0] = 0;
  sa.grid[1] = g.splitk;
  sa.grid[2] = g.prefill;
  sa.ws = W;
  sa.status_dev = status_dev;

  AttnArgs aa{};
  aa.q = (const __nv_bfloat16*)q;
  aa.q_rs = q_rs;
  aa.q_hs = q_hs;
  aa.k = (const __nv_bfloat16*)k;
  aa.v = (const __nv_bfloat16*)v;
  aa.rows = rows;
  aa.cols = cols;
  aa.Hkv = Hkv;
  aa.Hq = Hq;
  aa.group = Hq / Hkv;
  aa.D = D;
  aa.causal = sa.causal;
  aa.window = window;
  aa.scale_log2 = scale * 1.4426950408889634f;
  aa.out = (__nv_bfloat16*)out;
  aa.o_rs = o_rs;
  aa.o_hs = o_hs;
  aa.T = T;
  aa.ws = W;
  aa.status_dev = status_dev;
  AppendArgs apw;
  if (ap) {
    apw = *ap;
    apw.segs = W.segs;
  }
  return launch_all(sa, aa, D, g, tm, ap ? &apw : nullptr, (cudaStream_t)stream);
}

}  // namespace sdpa

using namespace sdpa;

extern "C" {

size_t sdpa_varlen_workspace_bytes(int64_t T, int Hq, int Hkv, int D, int S) {
  if (T < 0 || S < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return 0;
  if (D != 64 && D != 128 && D != 256) return 0;
  DevInfo di;
  Grids g;
  if (device_info(&di) == SDPA_OK) {
    g = grids_for(di, D);
  } else {
    g.splitk = 4096;  // no device: a bound above any real grid
    g.prefill = 1024;
    g_err[0] = 0;
  }
  return layout_workspace(nullptr, T, Hq, Hkv, D, S, g.splitk, g.prefill, nullptr);
}

sdpa_status sdpa_varlen(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                        int64_t q_head_stride, const void* k_store, const void* v_store,
                        int64_t rows, int cols, int Hkv, const int32_t* seq_info, int S,
                        int causal, int window, float scale, void* out, int64_t o_row_stride,
                        int64_t o_head_stride, void* workspace, size_t ws_bytes,
                        int32_t* status_dev, void* stream) {
  return run(q, T, Hq, D, q_row_stride, q_head_stride, k_store, v_store, rows, cols, Hkv, seq_info,
             S, nullptr, causal, window, scale, out, o_row_stride, o_head_stride, workspace,
             ws_bytes, status_dev, stream);
}

sdpa_status sdpa_varlen_append(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                               int64_t q_head_stride, const void* k_new, const void* v_new,
                               int64_t new_row_stride, int64_t new_head_stride, void* k_store,
                               void* v_store, int64_t rows, int cols, int Hkv, const int32_t* seq_info,
                               int S, int causal, int window, float scale, void* out,
                               int64_t o_row_stride, int64_t o_head_stride, void* workspace,
                               size_t ws_bytes, int32_t* status_dev, void* stream) {
  g_err[0] = 0;
  if (!k_new || !v_new) return fail(SDPA_ERR_NULL, "k_new or v_new is NULL");
  if (!aligned16(k_new) || !aligned16(v_new)) return fail(SDPA_ERR_ALIGN, "k_new and v_new must be 16-byte aligned");
  if (new_row_stride < 0 || new_head_stride < 0 || (new_row_stride % 8) || (new_head_stride % 8))
    return fail(SDPA_ERR_STRIDE, "new-row strides must be non-negative multiples of 8 elements");
  AppendArgs ap{};
  ap.k_new = (const __nv_bfloat16*)k_new;
  ap.v_new = (const __nv_bfloat16*)v_new;
  ap.new_rs = new_row_stride;
  ap.new_hs = new_head_stride;
  ap.k_store = (__nv_bfloat16*)k_store;
  ap.v_store = (__nv_bfloat16*)v_store;
  ap.rows = rows;
  ap.cols = cols;
  ap.Hkv = Hkv;
  ap.D = D;
  return run(q, T, Hq, D, q_row_stride, q_head_stride, k_store, v_store, rows, cols, Hkv, seq_info,
             S, nullptr, causal, window, scale, out, o_row_stride, o_head_stride, workspace,
             ws_bytes, status_dev, stream, &ap);
}

sdpa_status sdpa_varlen_modes(const void* q, int64_t T, int Hq, int D, int64_t q_row_stride,
                              int64_t q_head_stride, const void* k_store, const void* v_store,
                              int64_t rows, int cols, int Hkv, const int32_t* seq_info,
                              const int32_t* seg_mode, int S, float scale, void* out,
                              int64_t o_row_stride, int64_t o_head_stride, void* workspace,
                              size_t ws_bytes, int32_t* status_dev, void* stream) {
  g_err[0] = 0;
  if (!seg_mode && S > 0) return fail(SDPA_ERR_NULL, "seg_mode is NULL");
  return run(q, T, Hq, D, q_row_stride, q_head_stride, k_store, v_store, rows, cols, Hkv, seq_info,
             S, nullptr, 1, 0, scale, out, o_row_stride, o_head_stride, workspace, ws_bytes,
             status_dev, stream, nullptr, seg_mode);
}

sdpa_status sdpa_seq_clone(void* k_store, void* v_store, int64_t rows, int cols, int Hkv, int D,
                           int src_col, int dst_col, int64_t n, void* stream) {
  g_err[0] = 0;
  if (!k_store || !v_store) return fail(SDPA_ERR_NULL, "a store pointer is NULL");
  if (!aligned16(k_store) || !aligned16(v_store)) return fail(SDPA_ERR_ALIGN, "stores must be 16-byte aligned");
  if (rows <= 0 || cols <= 0 || Hkv <= 0 || n < 0)
    return fail(SDPA_ERR_SHAPE, "bad sizes: rows=%lld cols=%d Hkv=%d n=%lld", (long long)rows, cols, Hkv,
                (long long)n);
  if (D != 64 && D != 128 && D != 256) return fail(SDPA_ERR_HEAD_DIM, "head dim %d not in {64,128,256}", D);
  if (src_col < 0 || src_col >= cols || dst_col < 0 || dst_col >= cols)
    return fail(SDPA_ERR_ARG, "columns %d -> %d outside [0, %d)", src_col, dst_col, cols);
  const int64_t m = std::min(n, rows);
  if (m == 0 || src_col == dst_col) return SDPA_OK;
  DevInfo di;
  sdpa_status st = device_info(&di);
  if (st) return st;
  CloneArgs ca{};
  ca.k_store = (__nv_bfloat16*)k_store;
  ca.v_store = (__nv_bfloat16*)v_store;
  ca.m = m;
  ca.cols = cols;
  ca.Hkv = Hkv;
  ca.D = D;
  ca.src_col = src_col;
  ca.dst_col = dst_col;
  const int64_t total = m * Hkv * (D / 8);
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>((int64_t)di.sms * 8, (total + 4 * kCloneThreads - 1) / (4 * kCloneThreads)));
  void* args[] = {(void*)&ca};
  cudaError_t e = cudaLaunchKernel(clone_kernel_ptr(), dim3((unsigned)blocks), dim3(kCloneThreads), args, 0,
                                   (cudaStream_t)stream);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "clone launch: %s", cudaGetErrorString(e));
  return SDPA_OK;
}

sdpa_status sdpa_causal_prefill(const void* q, const void* k, const void* v, int64_t Lq,
                                int64_t Lkv, int Hq, int Hkv, int D, float scale, void* out,
                                void* workspace, size_t ws_bytes, void* stream) {
  g_err[0] = 0;
  if (Lq < 0 || Lkv <= 0) return fail(SDPA_ERR_SHAPE, "Lq=%lld Lkv=%lld", (long long)Lq, (long long)Lkv);
  if (Lq > INT32_MAX || Lkv > INT32_MAX) return fail(SDPA_ERR_SHAPE, "Lq or Lkv beyond 2^31-1");
  const int32_t seg[4] = {0, (int32_t)Lq, 0, (int32_t)Lkv};
  const int64_t rs = (int64_t)Hq * D;
  return run(q, Lq, Hq, D, rs, D, k, v, Lkv, 1, Hkv, nullptr, 1, seg, 1, 0, scale, out, rs, D,
             workspace, ws_bytes, nullptr, stream);
}

int sdpa_prefill_available(int D) {
  g_err[0] = 0;
  if (D != 64 && D != 128 && D != 256) {
    fail(SDPA_ERR_HEAD_DIM, "head dim %d not in {64,128,256}", D);
    return -1;
  }
  DevInfo di;
  if (device_info(&di) != SDPA_OK) return -1;
  return di.prefill_ok[d_index(D)] ? 1 : 0;
}

sdpa_status sdpa_set_route_policy(int policy) {
  if (policy != SDPA_ROUTE_AUTO && policy != SDPA_ROUTE_SPLITK && policy != SDPA_ROUTE_PREFILL)
    return fail(SDPA_ERR_ARG, "unknown route policy %d", policy);
  g_policy.store(policy);
  return SDPA_OK;
}

sdpa_status sdpa_set_timing_events(void* const* events, int n) {
  if (!events) {
    g_ev_on = false;
    return SDPA_OK;
  }
  if (n != 5) return fail(SDPA_ERR_ARG, "timing hook takes 5 events, got %d", n);
  for (int i = 0; i < 5; ++i) {
    if (!events[i]) return fail(SDPA_ERR_NULL, "timing event %d is NULL", i);
    g_ev[i] = (cudaEvent_t)events[i];
  }
  g_ev_on = true;
  return SDPA_OK;
}

sdpa_status sdpa_workspace_status(const void* workspace, size_t ws_bytes, int32_t* status_host, void* stream) {
  g_err[0] = 0;
  if (!workspace || !status_host) return fail(SDPA_ERR_NULL, "workspace or status_host is NULL");
  if ((uintptr_t)workspace % 256) return fail(SDPA_ERR_ALIGN, "workspace must be 256-byte aligned");
  if (ws_bytes < sizeof(SchedHdr)) return fail(SDPA_ERR_WORKSPACE, "workspace of %zu bytes has no header", ws_bytes);
  // the header opens every workspace layout; its status word is rewritten by each call's
  // scheduler and ORed by the attention kernels (SDPA_DEV_TIMEOUT)
  const SchedHdr* h = reinterpret_cast<const SchedHdr*>(workspace);
  int64_t v = 0;
  cudaStream_t st = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(&v, &h->status, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(SDPA_ERR_CUDA, "status read-back: %s", cudaGetErrorString(e));
  *status_host = (int32_t)v;
  return SDPA_OK;
}

const char* sdpa_last_error(void) { return g_err; }

int sdpa_version(void) { return 100; }

}  // extern "C"
