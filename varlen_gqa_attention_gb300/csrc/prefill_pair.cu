// prefill_pair.cu - tensor-memory attention kernel for long segments at D = 64 and 128 on
// sm_103a: two 128-row query tiles per CTA share every K/V tile.
//
// "[CUDA] Use Triton TMA for long-context causal prefill" (Summary: TMA-staged tiles,
// per-head-dim tile configurations, guarded online softmax so fully masked rows stay finite,
// real output strides) and "[executorch][cuda] Add a length-aware Triton SDPA over
// per-sequence KV columns" (segments over a column store, ring layers, causal / window
// masks, GQA).  The pages' Triton design targets SM90 / RTX 5090; this kernel is written
// for Blackwell's fifth-generation tensor cores:
//
//   * a persistent grid of one CTA per SM walks the stream-K tile line of the prefill route
//     (the scheduler's units are (segment, KV head, 256 packed rows r = i * group + g): the
//     query heads that share a KV head fill the MMA's M dimension together, GQA packing);
//     a unit is two halves of 128 rows, each with its own accumulators, so one K/V tile
//     feeds 256 rows and the K/V bytes read from L2 per flop halve against 128-row units;
//   * two producer warps move Q (both halves) and K tiles, and V tiles, with TMA (128-byte
//     swizzle) into rings of shared-memory stages; a tile whose store rows would wrap around
//     a ring store is never formed (the key range is tiled in two parts at the wrap), so
//     every tile is one box of the 4-d store tensor [rows, cols, Hkv, D];
//   * tensor memory (512 columns): S_h (fp32, 128 keys) for each half h, the softmax's P_h
//     written as bf16 pairs over the first 64 columns of S_h, and the output accumulators
//     O_0, O_1 (D columns each);
//   * the MMA warp issues tcgen05.mma (the whole warp runs the loop, one elected lane
//     issues) in the order S_0(0) S_1(0) | PV_0(0) S_0(1) PV_1(0) S_1(1) | PV_0(1) ...:
//     while one half's softmax works on its scores the tensor pipe computes the other
//     half's PV and next scores.  S_h(j+1) overwrites the columns PV_h(j) reads P_h(j)
//     from; tcgen05.mma operations of one thread execute in issue order, so it is issued
//     right behind PV_h(j) without a wait.  Completion is signalled with tcgen05.commit;
//   * one softmax warpgroup per half, one thread per row (= tensor-memory lane): the thread
//     reads its 128 scores, masks them by select (causal, window, the tile's end), keeps a
//     base-2 running max with lazy rescaling (O_h is rescaled, after PV_h(j-1) has landed,
//     only when the row max grows by more than 2^8), writes P_h and, at the end of a piece,
//     normalises O_h into `out` (the unit's only CTA) or writes a partial slot for the
//     combine pass.  No row is shared between threads, so the warpgroups never synchronise
//     with each other;
//   * V rows past the last visible key of a tile are zeroed in shared memory before the PV
//     MMA (rows past the end of a ring are zero-filled by TMA), so stale or NaN store cells
//     never meet a zero probability (0 * NaN).
// Every mbarrier wait is bounded; a wait that gives up sets SDPA_DEV_TIMEOUT, the roles stop
// issuing work, the producers wait (bounded) for the copies they issued, the MMA warp for
// its MMAs, and the CTA frees its tensor memory and exits.
#include <cuda.h>

#include "tc.cuh"

namespace sdpa {

template <int D>
struct PpCfg {
  static constexpr int BM = kPrefillRows;  // rows per half
  static constexpr int BN = kPrefillTile;  // keys per tile
  // K(j+1) is loaded once S(j-1) is done and V(j+1) once PV(j-2) is done, so each has more
  // than a tile's time to land
  static constexpr int KSTAGES = D == 64 ? 6 : 2;
  static constexpr int VSTAGES = D == 64 ? 6 : 3;
  static constexpr int NREG = D / 64;      // 64-element (128-byte) column regions
  static constexpr int QH_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int O_COL = 2 * BN;     // O_h at O_COL + h * D
  static constexpr int TMEM_COLS = 512;
  static constexpr int THREADS = 32 * 11;  // 2 softmax warpgroups + K and V producers + MMA
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * QH_BYTES;
  static constexpr int OFF_V = OFF_K + KSTAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + VSTAGES * KV_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
};
static_assert(PpCfg<64>::SMEM <= 232448 && PpCfg<128>::SMEM <= 232448, "pair prefill shared memory");
static_assert(PpCfg<64>::O_COL + 2 * 64 <= 512 && PpCfg<128>::O_COL + 2 * 128 <= 512, "pair prefill tensor memory");

// barrier slots (8 bytes each) inside the 512-byte barrier block
struct PpBars {
  static constexpr int kMaxStages = 6;
  static constexpr int K_FULL = 0;    // [6] K landed
  static constexpr int K_EMPTY = 6;   // [6] both halves' S of this stage's tile done
  static constexpr int V_FULL = 12;   // [6] V landed
  static constexpr int V_READY = 18;  // [6] V landed and, on a short tile, its tail zeroed
  static constexpr int V_EMPTY = 24;  // [6] both halves' PV of this stage's tile done
  static constexpr int S_FULL = 30;   // [2] S_h(j) computed
  static constexpr int P_FULL = 32;   // [2] the 128 rows of half h wrote P_h(j)
  static constexpr int PV_DONE = 34;  // [2] PV_h(j) done (O_h complete up to tile j)
  static constexpr int Q_FULL = 36;
  static constexpr int Q_EMPTY = 37;  // every S of the piece done: Q may be overwritten
  static constexpr int DRAIN = 38;
};
static_assert(PpCfg<64>::KSTAGES <= PpBars::kMaxStages && PpCfg<64>::VSTAGES <= PpBars::kMaxStages,
              "K/V ring deeper than the barrier arrays");

struct PpPiece {
  UnitRec ur;
  KeyTiles kt;
  int64_t ta, tb;
  int slot;
  bool has1;  // the unit has rows in its second half
};

__device__ __forceinline__ bool pp_next(PieceWalk& w, PpPiece& pc, int64_t rows) {
  if (!walk_next(w, pc.ur, pc.ta, pc.tb)) return false;
  pc.kt = key_tiles(pc.ur.lo, pc.ur.hi, rows, kPrefillTile);
  pc.slot = (int)(blockIdx.x - pc.ur.g_first);
  pc.has1 = pc.ur.rows > kPrefillRows;
  return true;
}

// 128 consecutive 32-bit columns of the warp's lanes: four loads, then one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, float* v) {
  uint32_t r[128];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%128];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%129];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%130];\n"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%131];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]),
        "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]),
        "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]),
        "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]),
        "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]),
        "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]),
        "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]),
        "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]),
        "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr), "r"(taddr + 32u), "r"(taddr + 64u), "r"(taddr + 96u)
      : "memory");
#pragma unroll
  for (int i = 0; i < 128; ++i) v[i] = __uint_as_float(r[i]);
}

// 16 columns of 32-bit words of the warp's lanes, without waiting for completion (the
// registers are read at issue; tmem_wait_st() waits for every such store of the thread).
__device__ __forceinline__ void tmem_st16u_nowait(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};\n" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// Packed two-lane fp32 arithmetic and three-input max (fewer issue slots for the softmax,
// which shares its schedulers with the producer and MMA warps).
__device__ __forceinline__ float pp_max3(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// (y0, y1) = (x0, x1) * a + c
__device__ __forceinline__ void pp_fma2(float& y0, float& y1, float x0, float x1, float a, float c) {
  asm("{\n .reg .b64 x, a, c, y;\n mov.b64 x, {%2, %3};\n mov.b64 a, {%4, %4};\n"
      " mov.b64 c, {%5, %5};\n fma.rn.f32x2 y, x, a, c;\n mov.b64 {%0, %1}, y;\n}\n"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a), "f"(c));
}
// (s0, s1) += (x0, x1)
__device__ __forceinline__ void pp_add2(float& s0, float& s1, float x0, float x1) {
  asm("{\n .reg .b64 s, x;\n mov.b64 s, {%0, %1};\n mov.b64 x, {%2, %3};\n"
      " add.rn.f32x2 s, s, x;\n mov.b64 {%0, %1}, s;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(x0), "f"(x1));
}

// What the softmax's tile loop of one piece needs (32-bit: key positions are below 2^31).
struct PpLoop {
  int32_t lo, wrap, hi, na;  // the unit's key tiling (KeyTiles)
  int32_t ta, n;             // the piece's first tile and its tile count
  int32_t rlo, rhi;          // the row's visible keys [rlo, rhi)
  uint32_t g;                // tiles of this half before the piece (barrier phases)
  uint32_t t_s, t_o;         // this row's S_h and O_h in tensor memory
  float sl2;                 // scale * log2(e)
  uint32_t bars;             // shared address of the barrier block
  int h;
};
struct PpLoopOut {
  float m, l;  // running max (base 2) and row sum
  bool ok;
};

// The softmax of one piece for one row of half h: per key tile, wait for S_h, read the row's
// 128 scores, mask, keep the running max (rescaling O_h lazily), write P_h and signal it.
template <int D>
__device__ __noinline__ PpLoopOut pp_softmax_tiles(const PpLoop lp, volatile int* abort) {
  constexpr int BN = kPrefillTile;
  const uint32_t b_s = lp.bars + 8u * (uint32_t)(PpBars::S_FULL + lp.h);
  const uint32_t b_p = lp.bars + 8u * (uint32_t)(PpBars::P_FULL + lp.h);
  const uint32_t b_pv = lp.bars + 8u * (uint32_t)(PpBars::PV_DONE + lp.h);
  PpLoopOut out;
  out.ok = true;
  float m_use = -INFINITY, l = 0.f;
  uint32_t g = lp.g;
  for (int j = 0; j < lp.n; ++j, ++g) {
    // the tile's first key and how many of its keys exist
    const int32_t t = lp.ta + j;
    const int32_t j0 = t < lp.na ? lp.lo + t * BN : lp.wrap + (t - lp.na) * BN;
    const int32_t valid = min(BN, (t < lp.na ? lp.wrap : lp.hi) - j0);
    const bool okw = __all_sync(0xffffffffu, mbar_wait(b_s, g & 1, abort));
    if (!okw) {
      out.ok = false;
      return out;
    }
    // this row's visible columns of the tile
    const int vlo = min(max(lp.rlo - j0, 0), valid);
    const int vhi = min(max(lp.rhi - j0, 0), valid);
    float x[BN];
    tc_fence_after();
    tmem_ld128(lp.t_s, x);
    // columns outside [vlo, vhi) (masked keys, cells past the tile's end) -> -inf
    if (vlo > 0 || vhi < BN) {
#pragma unroll
      for (int k = 0; k < BN; ++k) x[k] = (k >= vlo && k < vhi) ? x[k] : -INFINITY;
    }
    float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int k = 4; k < BN; k += 2) mx4[(k >> 1) & 3] = pp_max3(mx4[(k >> 1) & 3], x[k], x[k + 1]);
    // scale is positive, so max(scale * s) = scale * max(s)
    const float mx = fmaxf(pp_max3(mx4[0], mx4[1], mx4[2]), mx4[3]) * lp.sl2;
    // lazy rescale: the running max moves only when a row's tile max exceeds it by 2^8; O_h
    // is rescaled below, after P_h is written (the scores' registers are free by then) and
    // before P_h is signalled (PV_h(j) accumulates into the rescaled O_h)
    const float m_new = fmaxf(m_use, mx);
    const bool resc = m_new > m_use + 8.f;  // false while nothing is visible
    const bool need_o = resc && j > 0 && m_use != -INFINITY;
    const float f = resc ? exp2_approx(m_use - m_new) : 1.f;  // 0 while m_use = -inf
    if (resc) {
      l *= f;
      m_use = m_new;
    }
    const float nmu = m_use == -INFINITY ? 0.f : -m_use;
    // p = 2^(scale*s - m) (masked columns give 0), row sum; P as bf16 pairs over S_h, in four
    // stores of 16 columns as they are ready (one wait for all of them)
    float sum4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t pw[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const int e = 32 * c + 2 * k;
        float a0, a1;
        pp_fma2(a0, a1, x[e], x[e + 1], lp.sl2, nmu);
        const float p0 = exp2_approx(a0), p1 = exp2_approx(a1);
        pp_add2(sum4[(2 * k) & 3], sum4[(2 * k + 1) & 3], p0, p1);
        pw[k] = pack_bf16x2(p0, p1);
      }
      tmem_st16u_nowait(lp.t_s + 16 * c, pw);
    }
    tmem_wait_st();
    l += (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
    if (__any_sync(0xffffffffu, need_o)) {
      // rescale this row of O_h once PV_h(j-1) has landed in it
      if (!__all_sync(0xffffffffu, mbar_wait(b_pv, (g - 1) & 1, abort))) {
        out.ok = false;
        return out;
      }
      tc_fence_after();
      const float fo = need_o ? f : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(lp.t_o + 32 * c, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] *= fo;
        tmem_st32(lp.t_o + 32 * c, o);
      }
    }
    tc_fence_before();
    mbar_arrive(b_p);
  }
  out.m = m_use;
  out.l = l;
  return out;
}

template <int D>
__global__ void __launch_bounds__(PpCfg<D>::THREADS, 1)
    sdpa_prefill_pair_kernel(const AttnArgs A, const __grid_constant__ CUtensorMap tmQ,
                             const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = PpCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  griddep_wait();  // the scheduler's output
  griddep_launch();
  {
    // no tiles for this CTA in any phase (or none on the route): the whole CTA leaves
    // before any set-up, after one round of header loads
    PieceWalk probe;
    walk_begin(probe, A.ws, kRoutePrefill);
    if (!walk_phase(probe)) return;
  }

  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sBar = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int W_PROD_K = 8, W_PROD_V = 9, W_MMA = 10;
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(bar(PpBars::K_FULL + s), 1);
      mbar_init(bar(PpBars::K_EMPTY + s), 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(bar(PpBars::V_FULL + s), 1);
      mbar_init(bar(PpBars::V_READY + s), 1);
      mbar_init(bar(PpBars::V_EMPTY + s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(PpBars::S_FULL + h), 1);
      mbar_init(bar(PpBars::P_FULL + h), 32 * 4);
      mbar_init(bar(PpBars::PV_DONE + h), 1);
    }
    mbar_init(bar(PpBars::Q_FULL), 1);
    mbar_init(bar(PpBars::Q_EMPTY), 1);
    mbar_init(bar(PpBars::DRAIN), 1);
    s_abort = 0;
    mbar_fence_init();
  }
  if (warp == W_MMA) {
    tmem_alloc(smem_u32(&s_tmem), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;

  if (warp == W_PROD_K || warp == W_PROD_V) {
    // ------------------------------------------------------------ TMA producers
    // One warp streams Q and K tiles, the other V tiles: K(j) is released as soon as both
    // halves' S(j) are done, so the K warp runs ahead while the V warp waits for PV.
    const bool is_k = warp == W_PROD_K;
    constexpr int NS_K = C::KSTAGES, NS_V = C::VSTAGES;
    PieceWalk wk;
    walk_begin(wk, A.ws, kRoutePrefill);
    PpPiece pc;
    uint32_t issued = 0;   // K (or V) tiles whose copies this warp started
    uint32_t q_issued = 0; // pieces whose Q copies this warp started
    bool ok = true;
    while (ok && pp_next(wk, pc, A.rows)) {
      const int hk = pc.ur.hk;
      if (is_k) {
        if (lane == 0) {
          ok = mbar_wait(bar(PpBars::Q_EMPTY), (q_issued & 1) ^ 1, abort);
          if (ok) {
            mbar_expect_tx(bar(PpBars::Q_FULL), (pc.has1 ? 2 : 1) * C::QH_BYTES);
            const int qrow = pc.ur.q_start + (int)(((int64_t)pc.ur.rb * (2 * C::BM)) / A.group);
            for (int h = 0; h < (pc.has1 ? 2 : 1); ++h)
#pragma unroll
              for (int c = 0; c < C::NREG; ++c)
                tma_load_3d(sQ + h * C::QH_BYTES + c * (C::BM * 128), &tmQ, bar(PpBars::Q_FULL), 64 * c,
                            hk * A.group, qrow + h * (C::BM / A.group));
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++q_issued;
      }
      const int n = (int)(pc.tb - pc.ta);
      for (int j = 0; ok && j < n; ++j) {
        int64_t j0;
        int valid;
        key_tile(pc.kt, pc.ta + j, C::BN, &j0, &valid);
        const int row0 = (int)(j0 % A.rows);
        if (is_k) {
          const int s = issued % NS_K;
          if (lane == 0) {
            ok = mbar_wait(bar(PpBars::K_EMPTY + s), ((issued / NS_K) & 1) ^ 1, abort);
            if (ok) {
              mbar_expect_tx(bar(PpBars::K_FULL + s), C::KV_BYTES);
#pragma unroll
              for (int c = 0; c < C::NREG; ++c)
                tma_load_4d(sK + s * C::KV_BYTES + c * (C::BN * 128), &tmK, bar(PpBars::K_FULL + s), 64 * c, hk,
                            pc.ur.col, row0);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (ok) ++issued;
          continue;
        }
        const int s = issued % NS_V;
        const uint32_t use = issued / NS_V;
        if (lane == 0) {
          ok = mbar_wait(bar(PpBars::V_EMPTY + s), (use & 1) ^ 1, abort);
          if (ok) {
            // a full tile needs no zeroing: V_READY goes ahead of the copy, so it is complete
            // whenever V_FULL is
            if (valid == C::BN) mbar_arrive(bar(PpBars::V_READY + s));
            mbar_expect_tx(bar(PpBars::V_FULL + s), C::KV_BYTES);
#pragma unroll
            for (int c = 0; c < C::NREG; ++c)
              tma_load_4d(sV + s * C::KV_BYTES + c * (C::BN * 128), &tmV, bar(PpBars::V_FULL + s), 64 * c, hk,
                          pc.ur.col, row0);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        ++issued;
        if (valid < C::BN) {
          // V rows past the tile's last key: wait for the tile, then zero them
          ok = __all_sync(0xffffffffu, mbar_wait(bar(PpBars::V_FULL + s), use & 1, abort));
          if (!ok) break;
          const int bytes = (C::BN - valid) * 128;
#pragma unroll
          for (int c = 0; c < C::NREG; ++c) {
            uint8_t* reg = smem + C::OFF_V + s * C::KV_BYTES + c * (C::BN * 128) + valid * 128;
            for (int o = lane * 16; o < bytes; o += 32 * 16) *reinterpret_cast<uint4*>(reg + o) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(PpBars::V_READY + s));
        }
      }
    }
    // drain: the copies this warp started must land before the CTA exits (immediate on the
    // normal path, where the MMA warp consumed every stage and Q tile); each wait is bounded
    // on its own
    if (lane == 0) {
      const uint32_t ns = is_k ? NS_K : NS_V;
      const uint32_t first = issued > ns ? issued - ns : 0u;
      for (uint32_t g = first; g < issued; ++g) {
        int own = 0;
        mbar_wait(bar((is_k ? PpBars::K_FULL : PpBars::V_FULL) + g % ns), (g / ns) & 1, &own);
      }
      if (is_k && q_issued > 0) {
        int own = 0;
        mbar_wait(bar(PpBars::Q_FULL), (q_issued - 1) & 1, &own);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; one elected lane issues each
    // MMA and commit.
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, C::BN, false, false);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
    constexpr int KS = D / 16, KP = C::BN / 16;  // k-steps of S and of PV
    PieceWalk wk;
    walk_begin(wk, A.ws, kRoutePrefill);
    PpPiece pc;
    uint32_t gk = 0, gv = 0;     // K and V tiles consumed by this CTA
    uint32_t gp[2] = {0, 0};     // tiles of each half (S_FULL / P_FULL / PV_DONE phases)
    uint32_t pi = 0;
    bool ok = true;
    // Descriptors differ only in their start-address field (bits 0-13, address / 16), so each
    // MMA's operands are a base descriptor plus a byte offset / 16.
    const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
    const uint64_t k_desc = sdesc_sw128(sK, 16, 1024);
    const uint64_t v_desc = sdesc_sw128(sV, C::BN * 128, 1024);
    auto issue_s = [&](int h, uint32_t g) {  // S_h = Q_h K(g)^T
      const uint64_t kd = k_desc + (uint64_t)(((g % C::KSTAGES) * C::KV_BYTES) >> 4);
      const uint64_t qd = q_desc + (uint64_t)((h * C::QH_BYTES) >> 4);
      const uint32_t d = tmem + h * C::BN;
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        const uint32_t off = ((k >> 2) * (C::BM * 128) + (k & 3) * 32) >> 4;
        const uint32_t offk = ((k >> 2) * (C::BN * 128) + (k & 3) * 32) >> 4;
        tc_mma_ss_w(d, qd + off, kd + offk, IDESC_QK, k > 0 ? 1u : 0u);
      }
      tc_commit_w(bar(PpBars::S_FULL + h));
    };
    auto issue_pv = [&](int h, uint32_t g, uint32_t acc0) {  // O_h (+)= P_h V(g)
      const uint64_t vd = v_desc + (uint64_t)(((g % C::VSTAGES) * C::KV_BYTES) >> 4);
      const uint32_t pa = tmem + h * C::BN, od = tmem + C::O_COL + h * D;
#pragma unroll
      for (int k = 0; k < KP; ++k)
        tc_mma_ts_w(od, pa + 8 * k, vd + (uint64_t)((k * 16 * 128) >> 4), IDESC_PV, k > 0 ? 1u : acc0);
      tc_commit_w(bar(PpBars::PV_DONE + h));
    };
    auto wait_all = [&](uint32_t b, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(b, parity, abort));
    };
    // V(j) (and, on a short tile, its zeroed tail) for PV(j); K(j+1) for S(j+1).  The barriers
    // a group of MMAs will need next are tested (non-blocking) right after the group before
    // it has been issued, so the test's latency hides behind the MMA issue, which waits for
    // room in the tensor pipe; a blocking wait runs only when a test came back negative.  So
    // the one wait left between two groups is the one for a half's P.
    auto v_short = [&](int64_t t) -> bool {
      int64_t j0;
      int valid;
      key_tile(pc.kt, t, C::BN, &j0, &valid);
      return valid < C::BN;
    };
    auto test_v = [&](uint32_t g, bool shortv) -> bool {
      const uint32_t vs = g % C::VSTAGES, vph = (g / C::VSTAGES) & 1;
      return mbar_test_wait(bar(PpBars::V_FULL + vs), vph) &&
             (!shortv || mbar_test_wait(bar(PpBars::V_READY + vs), vph));
    };
    auto wait_v = [&](uint32_t g, bool shortv) -> bool {
      const uint32_t vs = g % C::VSTAGES, vph = (g / C::VSTAGES) & 1;
      return wait_all(bar(PpBars::V_FULL + vs), vph) && (!shortv || wait_all(bar(PpBars::V_READY + vs), vph));
    };
    auto test_k = [&](uint32_t g) -> bool {
      return mbar_test_wait(bar(PpBars::K_FULL + g % C::KSTAGES), (g / C::KSTAGES) & 1);
    };
    auto wait_k = [&](uint32_t g) -> bool {
      return wait_all(bar(PpBars::K_FULL + g % C::KSTAGES), (g / C::KSTAGES) & 1);
    };
    while (ok && pp_next(wk, pc, A.rows)) {
      const int n = (int)(pc.tb - pc.ta);
      const int nh = pc.has1 ? 2 : 1;
      ok = wait_all(bar(PpBars::Q_FULL), pi & 1) && wait_k(gk);
      if (!ok) break;
      tc_fence_after();
      for (int h = 0; h < nh; ++h) issue_s(h, gk);
      tc_commit_w(bar(PpBars::K_EMPTY + gk % C::KSTAGES));
      if (n == 1) tc_commit_w(bar(PpBars::Q_EMPTY));
      ok = wait_v(gv, v_short(pc.ta));
      if (!ok) break;
      bool next_short = n > 1 && v_short(pc.ta + 1);
      for (int j = 0; j < n; ++j) {
        const bool more = j + 1 < n;
        // half 0: PV_0(j) once P_0(j) is written, then S_0(j+1) over the same columns
        ok = wait_all(bar(PpBars::P_FULL + 0), gp[0] & 1);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, gv, j > 0 ? 1u : 0u);
        // tested while the PV MMAs queue: K(j+1), P_1(j), and with one half V(j+1)
        const bool ready_k = !more || test_k(gk + 1);
        const bool ready_p1 = nh == 1 || mbar_test_wait(bar(PpBars::P_FULL + 1), gp[1] & 1);
        bool ready_v = !more || nh == 2 || test_v(gv + 1, next_short);
        if (more) {
          if (!__all_sync(0xffffffffu, ready_k)) {
            ok = wait_k(gk + 1);
            if (!ok) break;
          }
          issue_s(0, gk + 1);
        }
        ++gp[0];
        if (nh == 2) {
          if (!__all_sync(0xffffffffu, ready_p1)) {
            ok = wait_all(bar(PpBars::P_FULL + 1), gp[1] & 1);
            if (!ok) break;
          }
          tc_fence_after();
          issue_pv(1, gv, j > 0 ? 1u : 0u);
          if (more) ready_v = test_v(gv + 1, next_short);  // tested while the PV MMAs queue
          if (more) issue_s(1, gk + 1);
          ++gp[1];
        }
        tc_commit_w(bar(PpBars::V_EMPTY + gv % C::VSTAGES));
        ++gv;
        if (more) {
          ++gk;
          tc_commit_w(bar(PpBars::K_EMPTY + gk % C::KSTAGES));
          if (j + 2 == n) tc_commit_w(bar(PpBars::Q_EMPTY));  // the piece's last S are issued
          if (!__all_sync(0xffffffffu, ready_v)) {  // the next tile's V
            ok = wait_v(gv, next_short);
            if (!ok) break;
          }
          next_short = j + 2 < n && v_short(pc.ta + j + 2);
        }
      }
      if (!ok) break;
      ++gk;
      ++pi;
    }
    // drain: wait (bounded) until every MMA this warp issued has finished
    tc_commit_w(bar(PpBars::DRAIN));
    int own = 0;
    mbar_wait(bar(PpBars::DRAIN), 0, &own);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Warpgroup h owns half h: thread = row = tensor-memory lane.  The tile loop of a piece
    // runs in pp_softmax_tiles (out of line, so that the walk and unit records stay in this
    // frame and only the loop's few values share the registers with a 128-key score row).
    const int h = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + h * C::BN;
    const uint32_t t_o = tmem + lane_off + C::O_COL + h * D;
    PieceWalk wk;
    walk_begin(wk, A.ws, kRoutePrefill);
    PpPiece pc;
    uint32_t g = 0;  // tiles of this half
    bool ok = true;
    while (ok && pp_next(wk, pc, A.rows)) {
      if (h == 1 && !pc.has1) continue;  // the unit has no second half
      const UnitRec& ur = pc.ur;
      const int rl = h * C::BM + row;  // row within the unit
      const bool live = rl < ur.rows;
      const int64_t r = (int64_t)ur.rb * (2 * C::BM) + rl;
      const int qi = (int)(r / A.group);
      PpLoop lp;
      lp.lo = (int32_t)pc.kt.lo;
      lp.wrap = (int32_t)pc.kt.wrap;
      lp.hi = (int32_t)pc.kt.hi;
      lp.na = (int32_t)pc.kt.na;
      lp.ta = (int32_t)pc.ta;
      lp.n = (int32_t)(pc.tb - pc.ta);
      lp.rlo = 1;  // padding rows see nothing
      lp.rhi = 0;
      if (live) {
        const RowWin w = row_window(qi, ur.q_len, ur.kv_end, ur.causal, ur.window);
        lp.rlo = w.lo;
        lp.rhi = w.hi;
      }
      lp.g = g;
      lp.t_s = t_s;
      lp.t_o = t_o;
      lp.sl2 = A.scale_log2;
      lp.bars = sBar;
      lp.h = h;
      const PpLoopOut lo = pp_softmax_tiles<D>(lp, abort);
      ok = lo.ok;
      if (!ok) break;
      g += lp.n;
      const float m_use = lo.m, l = lo.l;
      // epilogue: once the piece's last PV_h is done, normalise (direct) or write a partial
      ok = __all_sync(0xffffffffu, mbar_wait(bar(PpBars::PV_DONE + h), (g - 1) & 1, abort));
      if (!ok) break;
      tc_fence_after();
      const bool direct = ur.nslots == 1;
      const int hq = ur.hk * A.group + (int)(r % A.group);
      __nv_bfloat16* orow = A.out + ((int64_t)ur.q_start + qi) * A.o_rs + (int64_t)hq * A.o_hs;
      const int64_t pidx = ur.slot_base + (int64_t)pc.slot * ur.rows + rl;
      float* prow = A.ws.part_o[kRoutePrefill] + pidx * D;
      // a row with no visible key has l = 0 and writes zeros (never 0 * O)
      const bool empty = !(l > 0.f);
      const float w = direct ? (empty ? 0.f : 1.f / l) : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(t_o + 32 * c, o);
        if (!live) continue;
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = empty ? 0.f : o[k] * w;
        if (direct) {
#pragma unroll
          for (int k = 0; k < 32; k += 8) {
            uint4 v;
            v.x = pack_bf16x2(o[k], o[k + 1]);
            v.y = pack_bf16x2(o[k + 2], o[k + 3]);
            v.z = pack_bf16x2(o[k + 4], o[k + 5]);
            v.w = pack_bf16x2(o[k + 6], o[k + 7]);
            *reinterpret_cast<uint4*>(orow + 32 * c + k) = v;
          }
        } else {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(prow + 32 * c + k) = make_float4(o[k], o[k + 1], o[k + 2], o[k + 3]);
        }
      }
      if (live && !direct) A.ws.part_ml[kRoutePrefill][pidx] = make_float2(m_use, l);
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0 && s_abort) {
    atomicOr((int*)&A.ws.hdr->status, SDPA_DEV_TIMEOUT);
    if (A.status_dev) atomicOr(A.status_dev, SDPA_DEV_TIMEOUT);
  }
  if (warp == W_MMA) tmem_dealloc(tmem, C::TMEM_COLS);
}

template __global__ void sdpa_prefill_pair_kernel<64>(const AttnArgs, const __grid_constant__ CUtensorMap,
                                                      const __grid_constant__ CUtensorMap,
                                                      const __grid_constant__ CUtensorMap);
template __global__ void sdpa_prefill_pair_kernel<128>(const AttnArgs, const __grid_constant__ CUtensorMap,
                                                       const __grid_constant__ CUtensorMap,
                                                       const __grid_constant__ CUtensorMap);

const void* prefill_pair_kernel_ptr(int D) {
  return D == 64 ? (const void*)sdpa_prefill_pair_kernel<64> : (const void*)sdpa_prefill_pair_kernel<128>;
}
int prefill_pair_smem_bytes(int D) { return D == 64 ? PpCfg<64>::SMEM : PpCfg<128>::SMEM; }
int prefill_pair_block_threads(int D) { return D == 64 ? PpCfg<64>::THREADS : PpCfg<128>::THREADS; }

}  // namespace sdpa
