// combine.cu - log-sum-exp merge of split partials, and zero rows.
//
// Runs only when the scheduler found work for it (combine_work); then one warp per
// (packed row t, query head h):
//   * t owned by no live segment (uncovered, or an overlapping segment) -> 0
//     ("[executorch][cuda] Add a length-aware Triton SDPA over per-sequence KV columns",
//     PR description: rows no segment covers are zeroed);
//   * the unit holding (t, h) had a single CTA, or is a split-K unit of at most kMergeRows
//     rows (its last CTA merged the slots) -> already written; skip;
//   * no keys at all -> 0 (finite output for fully masked rows, "[CUDA] Use Triton TMA for
//     long-context causal prefill", Summary);
//   * otherwise merge the unit's slots: M = max m_c, L = sum l_c 2^(m_c - M),
//     O = sum o_c 2^(m_c - M) / L (m in base-2 units), L = 0 -> 0; round to bf16.
#include "common.cuh"

namespace sdpa {

constexpr int kCombineThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) sdpa_combine_kernel(AttnArgs A) {
  constexpr int PER = D / 32;  // elements per lane
  const int64_t gw = ((int64_t)blockIdx.x * kCombineThreads + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  griddep_wait();  // the attention kernels' slots and direct writes
  if (!A.ws.hdr->combine_work || gw >= A.T * A.Hq) return;
  const int64_t t = gw / A.Hq;
  const int h = (int)(gw % A.Hq);
  __nv_bfloat16* dst = A.out + t * A.o_rs + (int64_t)h * A.o_hs + lane * PER;
  const Workspace& W = A.ws;

  bool zero = true;
  const int s = W.row_seg[t];
  if (s >= 0) {
    const SegRec sg = W.segs[s];
    const int q = sg.route;
    if (q != kRouteNone) {
      const int rpu = q == kRoutePrefill ? kPrefillRows : kSplitkRows;
      const int64_t i = t - sg.q_start;
      const int hk = h / A.group;
      const int64_t r = i * A.group + (h % A.group);
      const int64_t rb = r / rpu;
      const int64_t u = (int64_t)sg.ubase[q] + (int64_t)hk * sg.nrb + rb;
      if (u < W.hdr->units[q]) {
        const UnitRec ur = W.units[q][u];
        // written by the unit's only CTA, or merged by the last of a split-K unit's CTAs
        if (ur.nslots == 1 || (q == kRouteSplitk && ur.nslots > 1 && ur.rows <= kMergeRows)) return;
        if (ur.nslots > 1) {
          zero = false;
          const int64_t rl = r - rb * rpu;
          const float2* ml = W.part_ml[q];
          const float* po = W.part_o[q];
          float M = -INFINITY;
          for (int c = lane; c < ur.nslots; c += 32)
            M = fmaxf(M, ml[ur.slot_base + (int64_t)c * ur.rows + rl].x);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
          const float Mu = M == -INFINITY ? 0.f : M;
          float L = 0.f, acc[PER];
#pragma unroll
          for (int k = 0; k < PER; ++k) acc[k] = 0.f;
          for (int c = 0; c < ur.nslots; ++c) {
            const int64_t pi = ur.slot_base + (int64_t)c * ur.rows + rl;
            const float2 v = ml[pi];
            const float f = exp2_approx(v.x - Mu);
            L += v.y * f;
            const float* src = po + pi * D + lane * PER;
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] += src[k] * f;
          }
          const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
          for (int k = 0; k < PER; k += 2)
            *reinterpret_cast<uint32_t*>(dst + k) = pack_bf16x2(acc[k] * inv, acc[k + 1] * inv);
        }
      }
    }
  }
  if (zero) {
#pragma unroll
    for (int k = 0; k < PER; k += 2) *reinterpret_cast<uint32_t*>(dst + k) = 0u;
  }
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
