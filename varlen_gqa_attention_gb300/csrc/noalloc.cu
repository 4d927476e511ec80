// noalloc.cu - an entry point for callers that cannot allocate device memory.
//
// sdpa_varlen needs a caller-provided workspace.  Some callers cannot provide one: code that
// runs where no allocator is available or allowed (a runtime with a fixed memory plan, a
// plugin that must not call cudaMalloc, a host language binding without a device allocator).
// sdpa_varlen_splitk_static serves them: it runs the scheduler, the split-K kernel and the
// combine pass (every segment on the split-K route) with their scratch in a file-scope
// device array of kStaticScratchBytes, and allocates nothing.
//
// The array is a host-side stand-in symbol in host code, not a device address: its device
// address is fetched with cudaGetSymbolAddress once per device (with that device current)
// on the first call there, and passed to the kernels.  That first call should come before
// any stream capture.  The address is kept for the life of the process: it assumes the
// device's primary context does too (after cudaDeviceReset it would be stale, so a caller
// that resets a device must not call this entry point on it again).  Every call on a device shares the one array, which keeps the last
// call's contents; nothing in it needs to start at zero (the scheduler kernel writes every
// field the later kernels read), but two calls that overlap on the GPU (different streams,
// or graphs replayed concurrently) race on it.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace sdpa {

constexpr size_t kStaticScratchBytes = (size_t)SDPA_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

namespace {

struct StaticDev {
  bool ready = false;
  void* scratch = nullptr;  // device address of g_static_scratch on this device
  int sms = 0;
  int per_sm[3] = {0, 0, 0};  // split-K CTAs per SM for D = 64, 128, 256
};
std::mutex g_static_mu;
StaticDev g_static_dev[64];
sdpa_status static_fail(sdpa_status code, const char* msg) {
  set_last_error(msg);
  return code;
}

int dix(int D) { return D == 64 ? 0 : D == 128 ? 1 : 2; }

// Once per device, with that device current: the scratch address and the launch facts.
sdpa_status static_setup(StaticDev* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return static_fail(SDPA_ERR_CUDA, "no current CUDA device");
  std::lock_guard<std::mutex> lk(g_static_mu);
  StaticDev& sd = g_static_dev[dev];
  if (!sd.ready) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return static_fail(SDPA_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
    }
    if (cudaDeviceGetAttribute(&sd.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return static_fail(SDPA_ERR_CUDA, "SM count query failed");
    if (cudaFuncSetAttribute(sched_kernel_ptr(), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sched_smem_bytes()) != cudaSuccess)
      return static_fail(SDPA_ERR_CUDA, "scheduler kernel setup failed");
    const int Ds[3] = {64, 128, 256};
    for (int k = 0; k < 3; ++k) {
      const void* f = splitk_kernel_ptr(Ds[k]);
      const int smem = splitk_smem_bytes(Ds[k]);
      int nb = 0;
      if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, f, kSplitkThreads, smem) != cudaSuccess)
        return static_fail(SDPA_ERR_CUDA, "split-K kernel setup failed");
      sd.per_sm[k] = nb > 0 ? nb : 1;
    }
    sd.scratch = p;
    sd.ready = true;
  }
  *out = sd;
  return SDPA_OK;
}

}  // namespace
}  // namespace sdpa

using namespace sdpa;

extern "C" sdpa_status sdpa_varlen_splitk_static(
    const void* q, int64_t T, int Hq, int D, int64_t q_row_stride, int64_t q_head_stride,
    const void* k_store, const void* v_store, int64_t rows, int cols, int Hkv, const int32_t* seq_info,
    int S, int causal, int window, float scale, void* out, int64_t o_row_stride, int64_t o_head_stride,
    int32_t* status_dev, void* stream) {
  set_last_error("");
  // the same argument checks, with the same messages, as sdpa_varlen
  sdpa_status st = check_common(T, Hq, Hkv, D, S, rows, cols, window, scale);
  if (st) return st;
  if ((st = check_tensors(q, k_store, v_store, out, seq_info, S, q_row_stride, q_head_stride, o_row_stride,
                          o_head_stride)))
    return st;

  StaticDev sd;
  if ((st = static_setup(&sd))) return st;
  // sdpa_varlen's workspace layout without the prefill route's tables.  The general grid if
  // its scratch fits; otherwise one CTA per SM (fewer partial slots).
  int64_t grid = (int64_t)sd.sms * sd.per_sm[dix(D)];
  size_t need = layout_workspace(nullptr, T, Hq, Hkv, D, S, grid, 0, nullptr, false);
  if (need > kStaticScratchBytes) {
    grid = sd.sms;
    need = layout_workspace(nullptr, T, Hq, Hkv, D, S, grid, 0, nullptr, false);
  }
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "these sizes need %zu bytes of scratch; the static scratch holds %zu bytes "
             "(use sdpa_varlen with a caller-provided workspace)",
             need, kStaticScratchBytes);
    return static_fail(SDPA_ERR_WORKSPACE, msg);
  }
  Workspace W;
  layout_workspace((char*)sd.scratch, T, Hq, Hkv, D, S, grid, 0, &W, false);

  SchedArgs sa{};
  sa.seq_info = seq_info;
  sa.S = S;
  sa.use_inline = 0;
  sa.T = T;
  sa.rows = rows;
  sa.cols = cols;
  sa.Hkv = Hkv;
  sa.group = Hq / Hkv;
  sa.causal = causal ? 1 : 0;
  sa.window = window;
  sa.D = D;
  sa.policy = SDPA_ROUTE_SPLITK;
  sa.prefill_ok = 0;
  sa.tile_pf = kPrefillTile;
  sa.grid[0] = 0;
  sa.grid[1] = grid;
  sa.grid[2] = 0;
  sa.ws = W;
  sa.status_dev = status_dev;

  AttnArgs aa{};
  aa.q = (const __nv_bfloat16*)q;
  aa.q_rs = q_row_stride;
  aa.q_hs = q_head_stride;
  aa.k = (const __nv_bfloat16*)k_store;
  aa.v = (const __nv_bfloat16*)v_store;
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
  aa.o_rs = o_row_stride;
  aa.o_hs = o_head_stride;
  aa.T = T;
  aa.ws = W;
  aa.status_dev = status_dev;

  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  e = launch_sched(sa, s);
  if (e == cudaSuccess) {
    void* args[] = {(void*)&aa};
    e = cudaLaunchKernel(splitk_kernel_ptr(D), dim3((unsigned)grid), dim3(kSplitkThreads), args,
                         splitk_smem_bytes(D), s);
  }
  if (e == cudaSuccess && T > 0) {
    void* args[] = {(void*)&aa};
    const int64_t blocks = std::min<int64_t>((T * Hq * 32 + 255) / 256, 8 * (int64_t)sd.sms);
    e = cudaLaunchKernel(combine_kernel_ptr(D), dim3((unsigned)blocks), dim3(256), args, 0, s);
  }
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "launch failed: %s", cudaGetErrorString(e));
    return static_fail(SDPA_ERR_CUDA, msg);
  }
  return SDPA_OK;
}

