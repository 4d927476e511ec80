// splitk.cu - split-K attention kernel for short steps (decode, draft blocks, small prefills).
//
// "[CUDA] Use Triton TMA for long-context causal prefill" (stack list: hardware-aware
// online-softmax split-K decode scheduling) and "[executorch][cuda] Add a length-aware Triton
// SDPA over per-sequence KV columns" (split-K for short steps).
//
// A persistent grid (a multiple of the SM count) walks the stream-K tile line the scheduler
// built: each CTA owns an equal share of key tiles across all units, a unit being
// (segment, KV head, up to 32 packed rows r = i * group + g).  Per unit and CTA:
//   * Q rows and 64-position K/V tiles are staged in shared memory with 16-byte cp.async
//     (coalesced: a store row of one KV head is D*2 contiguous bytes, fetched from DRAM as
//     one 256-byte block; ring rows wrap per row) through a three-stage ring (two at
//     D = 256), so two tiles stream in while one is used; two CTAs share an SM at D <= 128;
//   * each warp takes a 16-row group and a slice of the tile: S = Q K^T and O += P V with
//     bf16 m16n8k16 tensor-core MMAs and fp32 accumulation; two row groups split the tile's
//     keys in halves, one row group (decode: q_len=1, group 8) in quarters, so no warp runs
//     a whole tile of these legacy MMAs;
//   * online softmax in base 2 with quad shuffles for the row max / sum, masks applied by
//     select (never by adding), fully masked rows kept finite;
//   * the warps' slices are merged through shared memory, then the CTA either writes `out`
//     (it is the unit's only CTA) or a partial (max, sum, unnormalised O) that the combine
//     pass merges (merging in this kernel, by the last of a unit's CTAs, put the merges on
//     the kernel's tail: a decode step's kernel took 36.9 us against 30.7 us without them,
//     and the step itself was 2 us slower).
#include "common.cuh"

namespace sdpa {

template <int D>
struct SplitkSmem {
  // key tiles in flight: 3 stages keep two tiles loading while one is used (two CTAs per
  // SM at D <= 128); D = 256 tiles are twice as large, so two stages
  static constexpr int kStages = D == 256 ? 2 : 3;
  static constexpr int kRowBytes = D * 2;
  static constexpr int kQBytes = kSplitkRows * kRowBytes;
  static constexpr int kTileBytes = kSplitkTile * kRowBytes;
  static constexpr int kBytes = kQBytes + 2 * kStages * kTileBytes;
};

// Per-thread cursor over the key tiles of one unit: each thread always copies the same
// 16-byte chunk column of rows n0, n0 + kRowStep, ... of a tile, so only the tile's first
// store row (kept modulo `rows` incrementally) changes from tile to tile.
template <int D>
struct KvCursor {
  static constexpr int CH = D / 8;                      // 16-byte chunks per store row
  static constexpr int kRowStep = kSplitkThreads / CH;  // rows one pass of the CTA covers
  static constexpr int kPasses = kSplitkTile / kRowStep;
  const __nv_bfloat16* kb;  // this thread's chunk column of (column, KV head), store row 0
  const __nv_bfloat16* vb;
  int64_t rstride;          // elements between store rows
  int rows;
  int row0;                 // store row of the next tile's first key
  int n0, c;

  __device__ __forceinline__ void init(const AttnArgs& A, const SegRec& sg, int hk, int64_t first_pos) {
    c = threadIdx.x % CH;
    n0 = threadIdx.x / CH;
    rstride = (int64_t)A.cols * A.Hkv * D;
    const int64_t off = ((int64_t)sg.col * A.Hkv + hk) * D + c * 8;
    kb = A.k + off;
    vb = A.v + off;
    rows = (int)A.rows;
    row0 = (int)(first_pos % A.rows);
  }
  // Issues the copies of the next tile (keys [0, valid) of it; the rest are zero-filled),
  // then advances to the following tile.
  __device__ __forceinline__ void load(int valid, char* sK, char* sV) {
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      const int n = n0 + i * kRowStep;
      const bool ok = n < valid;
      int phys = row0 + n;
      if (phys >= rows) phys -= rows;  // valid keys span at most `rows` store rows
      const int64_t off = ok ? (int64_t)phys * rstride : 0;
      const uint32_t so = swz(n, c, D * 2);
      cp_async_16_row(smem_u32(sK + so), kb + off, ok);
      cp_async_16_row(smem_u32(sV + so), vb + off, ok);
    }
    row0 += kSplitkTile;
    if (row0 >= rows) row0 %= rows;
  }
};

// One warp's share of a unit: 16 packed rows x a slice of each key tile.
// s_count: [0] the done count of the CTA's previous piece, not yet counted (or null); [1] this
// piece's (null when it writes `out` directly).
template <int D, int NCS>
__device__ __forceinline__ void splitk_unit(const AttnArgs& A, const UnitRec& ur, const SegRec& sg,
                                            int64_t ta, int64_t tb, int slot, char* smem, float2* s_ml,
                                            int32_t** s_count) {
  using S = SplitkSmem<D>;
  constexpr int RB = S::kRowBytes;
  constexpr int SW = kSplitkTile / NCS;  // keys per warp slice
  constexpr int NB = SW / 8;             // n8 blocks per slice
  constexpr int ND = D / 8;              // n8 blocks of the output
  char* sQ = smem;
  char* sK = smem + S::kQBytes;
  constexpr int kStages = S::kStages;
  char* sV = sK + kStages * S::kTileBytes;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mt = warp / NCS, cs = warp % NCS;
  const int gq = lane >> 2, tq = lane & 3;
  const int R = ur.rows;
  const int64_t r0 = (int64_t)ur.rb * kSplitkRows;

  // key positions of this CTA's share of the unit
  const int64_t pos_lo = (int64_t)ur.lo + ta * kSplitkTile;
  const int64_t pos_hi = min((int64_t)ur.lo + tb * kSplitkTile, (int64_t)ur.hi);
  const int ntiles = (int)(tb - ta);

  // Q rows (packed r -> query row i = r / group, head hk*group + r % group)
  {
    constexpr int CH = D / 8;
    for (int idx = tid; idx < kSplitkRows * CH; idx += kSplitkThreads) {
      const int rl = idx / CH, c = idx % CH;
      const bool ok = rl < R;
      int64_t off = 0;
      if (ok) {
        const int64_t r = r0 + rl;
        const int64_t i = r / A.group;
        const int h = ur.hk * A.group + (int)(r % A.group);
        off = (sg.q_start + i) * A.q_rs + (int64_t)h * A.q_hs + c * 8;
      }
      cp_async_16(smem_u32(sQ + swz(rl, c, RB)), A.q + off, ok);
    }
  }
  // prologue: Q and the first kStages-1 tiles, one commit group per tile (empty past the end)
  KvCursor<D> cur;
  cur.init(A, sg, ur.hk, pos_lo);
  for (int st = 0; st < kStages - 1; ++st) {
    if (st < ntiles)
      cur.load((int)min((int64_t)kSplitkTile, pos_hi - pos_lo - (int64_t)st * kSplitkTile),
               sK + st * S::kTileBytes, sV + st * S::kTileBytes);
    cp_async_commit();
  }

  // this thread's two rows: local rows mt*16 + gq and +8
  int32_t rlo[2], rhi[2];
  bool live[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int rl = mt * 16 + gq + 8 * e;
    live[e] = rl < R;
    if (live[e]) {
      const int i = (int)((r0 + rl) / A.group);
      RowWin w = row_window(i, sg.q_len, sg.kv_end, sg.causal, sg.window);
      rlo[e] = (int32_t)max((int64_t)w.lo, pos_lo);
      rhi[e] = (int32_t)min((int64_t)w.hi, pos_hi);
    } else {
      rlo[e] = INT32_MIN;  // padding rows: never stored, Q = 0 keeps them finite
      rhi[e] = INT32_MAX;
    }
  }
  const int32_t lo_max = max(rlo[0], rlo[1]), hi_min = min(rhi[0], rhi[1]);

  float o[ND][4];
#pragma unroll
  for (int nd = 0; nd < ND; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const float sl2 = A.scale_log2;

  for (int kt = 0; kt < ntiles; ++kt) {
    // tile kt + kStages - 1 goes into the stage tile kt - 1 used (freed by the barrier that
    // ended the previous iteration); then wait until tile kt has landed
    if (kt + kStages - 1 < ntiles) {
      const int st = (kt + kStages - 1) % kStages;
      cur.load((int)min((int64_t)kSplitkTile, pos_hi - pos_lo - (int64_t)(kt + kStages - 1) * kSplitkTile),
               sK + st * S::kTileBytes, sV + st * S::kTileBytes);
    }
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    __syncthreads();
    const char* cK = sK + (kt % kStages) * S::kTileBytes;
    const char* cV = sV + (kt % kStages) * S::kTileBytes;
    const int64_t tile0 = pos_lo + (int64_t)kt * kSplitkTile + cs * SW;  // first key of slice

    // S = Q K^T over the slice
    float s[NB][4];
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) s[nb][0] = s[nb][1] = s[nb][2] = s[nb][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a[4];
      ldmatrix_x4(smem_u32(sQ + swz(mt * 16 + (lane & 15), kk * 2 + (lane >> 4), RB)), a[0], a[1],
                  a[2], a[3]);
#pragma unroll
      for (int nb = 0; nb < NB; nb += 2) {
        uint32_t b0, b1, b2, b3;
        const int pos = cs * SW + nb * 8 + (lane & 7) + ((lane >> 4) << 3);
        ldmatrix_x4(smem_u32(cK + swz(pos, kk * 2 + ((lane >> 3) & 1), RB)), b0, b1, b2, b3);
        mma_bf16_16816(s[nb], a, b0, b1);
        mma_bf16_16816(s[nb + 1], a, b2, b3);
      }
    }

    // mask (select, on the raw scores), online softmax in base 2 with a lazily updated max:
    // O and l are only rescaled when a row's max grows by more than 2^8
    const bool full = tile0 >= lo_max && tile0 + SW <= hi_min;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int rr = e >> 1;
        float x = s[nb][e];
        if (!full) {
          const int64_t j = tile0 + nb * 8 + 2 * tq + (e & 1);
          const bool vis = !live[rr] || (j >= rlo[rr] && j < rhi[rr]);
          // padding rows: keys past the share are zero-filled, harmless
          x = vis ? x : -INFINITY;
        }
        s[nb][e] = x;
        mx[rr] = fmaxf(mx[rr], x);
      }
    }
    float alpha[2], nmu[2];
    bool resc = false;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 1));
      mx[rr] = fmaxf(mx[rr], __shfl_xor_sync(0xffffffffu, mx[rr], 2));
      const float mn = fmaxf(m[rr], mx[rr] * sl2);  // scale > 0: max(scale*s) = scale*max(s)
      const bool up = mn > m[rr] + 8.f;            // false while nothing is visible
      alpha[rr] = up ? exp2_approx(m[rr] - mn) : 1.f;
      if (up) m[rr] = mn;
      resc |= up;
      nmu[rr] = m[rr] == -INFINITY ? 0.f : -m[rr];
    }
    float ls[2] = {0.f, 0.f};
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float p = exp2_approx(fmaf(s[nb][e], sl2, nmu[e >> 1]));
        s[nb][e] = p;
        ls[e >> 1] += p;
      }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) l[rr] = l[rr] * alpha[rr] + ls[rr];
    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
      for (int nd = 0; nd < ND; ++nd) {
        o[nd][0] *= alpha[0];
        o[nd][1] *= alpha[0];
        o[nd][2] *= alpha[1];
        o[nd][3] *= alpha[1];
      }
    }

    // O += P V
#pragma unroll
    for (int k2 = 0; k2 < SW / 16; ++k2) {
      uint32_t a[4];
      a[0] = pack_bf16x2(s[2 * k2][0], s[2 * k2][1]);
      a[1] = pack_bf16x2(s[2 * k2][2], s[2 * k2][3]);
      a[2] = pack_bf16x2(s[2 * k2 + 1][0], s[2 * k2 + 1][1]);
      a[3] = pack_bf16x2(s[2 * k2 + 1][2], s[2 * k2 + 1][3]);
      const int pos = cs * SW + k2 * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int nd = 0; nd < ND; nd += 2) {
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4_trans(smem_u32(cV + swz(pos, nd + (lane >> 4), RB)), b0, b1, b2, b3);
        mma_bf16_16816(o[nd], a, b0, b1);
        mma_bf16_16816(o[nd + 1], a, b2, b3);
      }
    }
    __syncthreads();
  }

  // row sums over the quad
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 1);
    l[rr] += __shfl_xor_sync(0xffffffffu, l[rr], 2);
  }

  // merge the warps' slices through shared memory (the K/V buffers are free now)
  float* mo = reinterpret_cast<float*>(sK);  // [4 warps][16 rows][D]
  {
    float* mw = mo + warp * 16 * D;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      const int d = nd * 8 + 2 * tq;
      *reinterpret_cast<float2*>(mw + gq * D + d) = make_float2(o[nd][0], o[nd][1]);
      *reinterpret_cast<float2*>(mw + (gq + 8) * D + d) = make_float2(o[nd][2], o[nd][3]);
    }
    if (tq == 0) {
      s_ml[warp * 16 + gq] = make_float2(m[0], l[0]);
      s_ml[warp * 16 + gq + 8] = make_float2(m[1], l[1]);
    }
  }
  __syncthreads();

  // the previous piece's partial slot, written a whole piece ago, is counted now: a release
  // waits for the CTA's earlier writes to land, which by now they have (counted at the end
  // of their own piece, it would wait on the slot just written, under full memory load)
  if (tid == 0 && s_count[0] != nullptr) {
    red_add_release(s_count[0], 1);
    s_count[0] = nullptr;
  }
  const bool direct = ur.nslots == 1;
  // the output row of local row rl, dims d0 .. d0 + 7, normalised by 1 / L (0 when L = 0)
  auto store_out = [&](int rl, int d0, const float* acc, float L) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int64_t r = r0 + rl;
    const int64_t i = r / A.group;
    const int h = ur.hk * A.group + (int)(r % A.group);
    uint4 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    pk.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
    pk.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(A.out + (sg.q_start + i) * A.o_rs + (int64_t)h * A.o_hs + d0) = pk;
  };
  for (int idx = tid; idx < R * (D / 8); idx += kSplitkThreads) {
    const int rl = idx / (D / 8), d0 = (idx % (D / 8)) * 8;
    const int mtr = rl / 16, rin = rl % 16;
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < NCS; ++c) M = fmaxf(M, s_ml[(mtr * NCS + c) * 16 + rin].x);
    const float Mu = M == -INFINITY ? 0.f : M;
    float L = 0.f, acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
    for (int c = 0; c < NCS; ++c) {
      const int w = mtr * NCS + c;
      const float2 ml = s_ml[w * 16 + rin];
      const float f = exp2_approx(ml.x - Mu);
      L += ml.y * f;
      const float* src = mo + (w * 16 + rin) * D + d0;
      const float4 u0 = *reinterpret_cast<const float4*>(src);
      const float4 u1 = *reinterpret_cast<const float4*>(src + 4);
      acc[0] += u0.x * f; acc[1] += u0.y * f; acc[2] += u0.z * f; acc[3] += u0.w * f;
      acc[4] += u1.x * f; acc[5] += u1.y * f; acc[6] += u1.z * f; acc[7] += u1.w * f;
    }
    if (direct) {
      store_out(rl, d0, acc, L);
    } else {
      const int64_t pi = ur.slot_base + (int64_t)slot * R + rl;
      if (d0 == 0) A.ws.part_ml[kRouteSplitk][pi] = make_float2(M, L);
      float* dst = A.ws.part_o[kRouteSplitk] + pi * D + d0;
      *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
  __syncthreads();
}

template <int D>
__global__ void __launch_bounds__(kSplitkThreads) sdpa_splitk_kernel(AttnArgs A) {
  extern __shared__ __align__(128) char smem[];
  __shared__ float2 s_ml[4 * 16];
  __shared__ int32_t* s_count[2];
  griddep_wait();    // the scheduler's output (and the prefill kernel's end)
  griddep_launch();
  PieceWalk wk;
  walk_begin(wk, A.ws, kRouteSplitk);  // no work on this route: the walk ends at once
  UnitRec ur;
  int64_t ta, tb;
  // Done counts (kept in shared memory, not in registers across a piece): the combine pass
  // merges a split unit as soon as all its CTAs have counted its slot, while other CTAs still
  // stream.  A piece's slot is counted in the next piece's epilogue, or as the CTA ends.
  if (threadIdx.x == 0) s_count[0] = nullptr;
  while (walk_next(wk, ur, ta, tb)) {
    SegRec sg;  // the unit record carries its segment's entry: no second dependent load
    sg.q_start = ur.q_start;
    sg.q_len = ur.q_len;
    sg.col = ur.col;
    sg.kv_end = ur.kv_end;
    sg.causal = ur.causal;
    sg.window = ur.window;
    const int slot = (int)(blockIdx.x - ur.g_first);
    // the walk has moved past the piece's unit
    if (threadIdx.x == 0) s_count[1] = ur.nslots > 1 ? A.ws.unit_done + (wk.u - 1) : nullptr;
    if (ur.rows <= 16)
      splitk_unit<D, 4>(A, ur, sg, ta, tb, slot, smem, s_ml, s_count);
    else
      splitk_unit<D, 2>(A, ur, sg, ta, tb, slot, smem, s_ml, s_count);
    if (threadIdx.x == 0) s_count[0] = s_count[1];
  }
  // the last piece ended on a barrier: its slot is complete (the release add is cumulative
  // over the CTA's writes before it)
  if (threadIdx.x == 0 && s_count[0] != nullptr) red_add_release(s_count[0], 1);
}

template __global__ void sdpa_splitk_kernel<64>(AttnArgs);
template __global__ void sdpa_splitk_kernel<128>(AttnArgs);
template __global__ void sdpa_splitk_kernel<256>(AttnArgs);

int splitk_smem_bytes(int D) {
  switch (D) {
    case 64: return SplitkSmem<64>::kBytes;
    case 128: return SplitkSmem<128>::kBytes;
    default: return SplitkSmem<256>::kBytes;
  }
}

const void* splitk_kernel_ptr(int D) {
  switch (D) {
    case 64: return (const void*)sdpa_splitk_kernel<64>;
    case 128: return (const void*)sdpa_splitk_kernel<128>;
    default: return (const void*)sdpa_splitk_kernel<256>;
  }
}

}  // namespace sdpa
