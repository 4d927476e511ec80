// combine.cu - log-sum-exp merge of split partials, and zero rows.
//
// Runs only when the scheduler found work for it (combine_work); then one warp per
// (packed row t, query head h), which finds the row's unit through the scheduler's row record:
//   * t owned by no live segment (uncovered, or an overlapping segment) -> 0
//     ("[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns",
//     PR description: rows no segment covers are zeroed);
//   * the unit holding (t, h) had a single CTA -> already written; skip;
//   * no keys at all -> 0 (finite output for fully masked rows, "[CUDA] Use Triton TMA for
//     long-context causal prefill", Summary);
//   * otherwise merge the unit's slots: M = max m_c, L = sum l_c 2^(m_c - M),
//     O = sum o_c 2^(m_c - M) / L (m in base-2 units, accumulated online over the slots, four
//     slots' loads in flight at a time), L = 0 -> 0; round to bf16.
// The pass does not wait for the attention kernels to finish: it is launched (programmatic
// dependent launch) once the split-K kernel has passed its own wait, i.e. once the scheduler
// and the prefill kernel have finished, and each warp waits only for its split-K unit's CTAs
// (the unit's done count reaches nslots; bounded, SDPA_DEV_TIMEOUT past two seconds).  Units
// that finish early are merged while the split-K kernel's last CTAs still stream.  The
// scheduler's records and the prefill kernel's slots come from grids that finished before
// this one was launched, so plain loads see them; the split-K slots are read after the
// acquire, through L2.
#include "common.cuh"

namespace sdpa {

constexpr int kCombineThreads = 256;

// Waits until *count reaches n (the unit's CTAs have written their slots); false after about
// two seconds.
__device__ __forceinline__ bool wait_done(const int32_t* count, int32_t n) {
  if (ld_acquire(count) >= n) return true;
  uint64_t t0;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t0));
  for (;;) {
    __nanosleep(200);
    if (ld_acquire(count) >= n) return true;
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    if (t - t0 > 2000000000ull) return false;
  }
}

// One warp: packed row t, query head h (gw = t * Hq + h).
template <int D>
__device__ __forceinline__ void combine_row(const AttnArgs& A, int64_t gw, int lane, int64_t U1, int64_t U2) {
  constexpr int PER = D / 32;  // elements per lane
  const int64_t t = gw / A.Hq;
  const int h = (int)(gw % A.Hq);
  __nv_bfloat16* dst = A.out + t * A.o_rs + (int64_t)h * A.o_hs + lane * PER;
  const Workspace& W = A.ws;
  const int4 ri = W.row_info[t];

  bool zero = true;
  const int q = ri.x;
  if (q != kRouteNone) {
    // route-indexed fields picked by select: a runtime index would copy them to local memory
    const bool pf = q == kRoutePrefill;
    const int rpu = pf ? prefill_unit_rows(D) : kSplitkRows;
    const int hk = h / A.group;
    const int64_t r = (int64_t)ri.w * A.group + (h % A.group);
    const int64_t rb = r / rpu;
    const int64_t u = (int64_t)ri.y + (int64_t)hk * ri.z + rb;
    if (u < (pf ? U2 : U1)) {
      const UnitRec ur = (pf ? W.units[kRoutePrefill] : W.units[kRouteSplitk])[u];
      if (ur.nslots == 1) return;  // written by the unit's only CTA
      if (ur.nslots > 1) {
        zero = false;
        if (!pf && !wait_done(W.unit_done + u, ur.nslots)) {
          if (lane == 0) {
            atomicOr((unsigned long long*)&W.hdr->status, (unsigned long long)SDPA_DEV_TIMEOUT);
            if (A.status_dev) atomicOr(A.status_dev, SDPA_DEV_TIMEOUT);
          }
          return;
        }
        // online log-sum-exp over the slots, four slots' loads in flight at a time:
        // M' = max(M, m_c), L' = L 2^(M - M') + l_c 2^(m_c - M'), O likewise
        const int64_t rl = r - rb * rpu;
        const float2* ml = (pf ? W.part_ml[kRoutePrefill] : W.part_ml[kRouteSplitk]) + ur.slot_base + rl;
        const float* po = (pf ? W.part_o[kRoutePrefill] : W.part_o[kRouteSplitk]) +
                          (ur.slot_base + rl) * D + lane * PER;
        const int64_t stride = ur.rows;  // partial rows between one slot and the next
        float M = -INFINITY, L = 0.f, acc[PER];
#pragma unroll
        for (int k = 0; k < PER; ++k) acc[k] = 0.f;
        constexpr int kBatch = 4;
        for (int c0 = 0; c0 < ur.nslots; c0 += kBatch) {
          float2 v[kBatch];
          float o[kBatch][PER];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            v[b] = make_float2(-INFINITY, 0.f);
            if (c0 + b < ur.nslots) {
              const int64_t c = c0 + b;
              v[b] = __ldcg(ml + c * stride);
              // PER = D / 32 floats per lane: 2, 4 or 8, so 8-byte loads at D = 64
              if constexpr (PER % 4 == 0) {
#pragma unroll
                for (int k = 0; k < PER; k += 4) {
                  const float4 u = __ldcg(reinterpret_cast<const float4*>(po + c * stride * D + k));
                  o[b][k] = u.x; o[b][k + 1] = u.y; o[b][k + 2] = u.z; o[b][k + 3] = u.w;
                }
              } else {
#pragma unroll
                for (int k = 0; k < PER; k += 2) {
                  const float2 u = __ldcg(reinterpret_cast<const float2*>(po + c * stride * D + k));
                  o[b][k] = u.x; o[b][k + 1] = u.y;
                }
              }
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if (v[b].x == -INFINITY) continue;  // an empty (or absent) slot adds nothing
            const float Mn = fmaxf(M, v[b].x);
            const float fo = exp2_approx(M - Mn), fc = exp2_approx(v[b].x - Mn);
            M = Mn;
            L = L * fo + v[b].y * fc;
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] = acc[k] * fo + o[b][k] * fc;
          }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int k = 0; k < PER; k += 2)
          *reinterpret_cast<uint32_t*>(dst + k) = pack_bf16x2(acc[k] * inv, acc[k + 1] * inv);
      }
    }
  }
  if (zero) {
#pragma unroll
    for (int k = 0; k < PER; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = 0u;
  }
}

// A grid of at most 8 CTAs per SM (a full SM's worth of warps) walks the (row, head) pairs,
// so that a call with many rows and nothing to merge does not pay for launching a CTA per 8
// pairs.
template <int D>
__global__ void __launch_bounds__(kCombineThreads) sdpa_combine_kernel(AttnArgs A) {
  const Workspace& W = A.ws;
  // independent loads, issued together: whether there is work and the routes' unit counts
  const int64_t work = W.hdr->combine_work;
  const int64_t U1 = W.hdr->units[kRouteSplitk], U2 = W.hdr->units[kRoutePrefill];
  if (!work) return;
  const int lane = threadIdx.x & 31;
  const int64_t n = A.T * A.Hq, stride = (int64_t)gridDim.x * (kCombineThreads / 32);
  for (int64_t gw = ((int64_t)blockIdx.x * kCombineThreads + threadIdx.x) >> 5; gw < n; gw += stride)
    combine_row<D>(A, gw, lane, U1, U2);
}

template __global__ void sdpa_combine_kernel<64>(AttnArgs);
template __global__ void sdpa_combine_kernel<128>(AttnArgs);
template __global__ void sdpa_combine_kernel<256>(AttnArgs);

const void* combine_kernel_ptr(int D) {
  switch (D) {
    case 64: return (const void*)sdpa_combine_kernel<64>;
    case 128: return (const void*)sdpa_combine_kernel<128>;
    default: return (const void*)sdpa_combine_kernel<256>;
  }
}

}  // namespace sdpa
