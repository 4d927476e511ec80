// prefill.cu - tensor-memory attention kernel for long segments on sm_103a at D = 256 (one
// 128-row query tile per CTA: its output accumulator alone takes half the tensor memory);
// D = 64 and 128 use the two-tile kernel of prefill_pair.cu.
//
// "[CUDA] Use Triton TMA for long-context causal prefill" (Summary: TMA-staged tiles,
// per-head-dim tile configurations, guarded online softmax so fully masked rows stay finite,
// real output strides) and "[executorch][cuda] Add a length-aware Triton SDPA over
// per-sequence KV columns" (segments over a column store, causal / window masks, GQA).
// The pages' Triton design targets SM90 / RTX 5090; this kernel is written for Blackwell's
// fifth-generation tensor cores instead:
//
//   * a persistent grid of one CTA per SM walks the stream-K tile line of the prefill route
//     (same scheduler output as the split-K kernel): every CTA gets the same number of key
//     tiles, units being (segment, KV head, 128 packed rows r = i * group + g) - the query
//     heads sharing a KV head fill the MMA's M dimension together (GQA packing);
//   * two producer warps move Q and K tiles, and V tiles, with TMA (128-byte swizzle) into
//     rings of shared-memory stages; the store is a 4-d tensor [rows, cols, Hkv, D], so a tile of one
//     column and KV head is one box (a key range that wraps around a ring store is tiled in
//     two parts at the wrap, so no tile's store rows wrap);
//   * the MMA warp issues tcgen05.mma (the whole warp runs the loop, one elected lane
//     issues): S = Q K^T into one of two tensor-memory buffers (fp32, 128 lanes x BN
//     columns) and O += P V with P read from tensor memory; S(g+2) goes out as soon as the
//     softmax has read S(g) out, PV(g) once P(g) is written; completion is signalled with
//     tcgen05.commit on mbarriers;
//   * two softmax warpgroups each take half of every tile's key columns, one thread per row
//     (= tensor-memory lane): the thread reads its S half-row, masks by select (causal,
//     window, the tile's end), keeps a base-2 running max shared by the two halves with lazy
//     rescaling (one barrier per tile checks that no row's tile max left the 2^8 window; only
//     then are maxima swapped and O rescaled) and writes P as bf16 pairs into tensor memory;
//     at the end of a piece the two row-sum halves are added and each warpgroup writes its
//     half of O's columns to `out` (the unit's only CTA) or to a partial for the combine pass;
//   * V rows past the last visible key of a unit are zeroed in shared memory before the PV
//     MMA, so stale or NaN store cells never meet a zero probability (0 * NaN).
// Every mbarrier wait is bounded; a wait that gives up sets SDPA_DEV_TIMEOUT and the CTA
// unwinds, frees its tensor memory and exits.
#include <cuda.h>

#include "tc.cuh"

namespace sdpa {

template <int D>
struct PfCfg {
  static constexpr int BM = kPrefillRows;                 // 128 packed rows
  static constexpr int BN = D == 256 ? 64 : kPrefillTile;  // keys per tile
  static constexpr int HALF = BN / 2;                     // key columns per softmax warpgroup
  static constexpr int STAGES = D == 64 ? 6 : (D == 128 ? 3 : 2);  // K/V ring depth
  static constexpr int NREG = D / 64;                     // 64-element (128-byte) column regions
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;             // K (or V) of one stage
  // Tensor memory: S_b fp32 [b*BN, (b+1)*BN); P_b as bf16 pairs [P_COL + b*BN/2, +BN/2);
  // one O accumulator of D columns.  Two softmax warpgroups split every tile's key columns.
  static constexpr int S_COL0 = 0;
  static constexpr int P_COL = 2 * BN;
  static constexpr int O_COL = D == 256 ? 256 : 3 * BN;
  static constexpr int TMEM_COLS = 512;
  static constexpr int SOFT_WARPS = 8;
  static constexpr int THREADS = 32 * (SOFT_WARPS + 3);  // + K and V producers + MMA issuer
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr int BAR_BYTES = 512;
  static constexpr int SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
};
static_assert(PfCfg<256>::STAGES <= 6, "K/V ring deeper than the barrier arrays");
static_assert(PfCfg<256>::SMEM <= 232448, "prefill D=256 shared memory");
static_assert(PfCfg<256>::O_COL + 256 <= 512 && PfCfg<256>::P_COL + 64 <= PfCfg<256>::O_COL,
              "prefill tensor-memory layout");

// barrier slots (8 bytes each) inside the barrier block
struct PfBars {
  // K and V stages are filled and released separately.  K(g) is free once S(g) is done:
  // the softmax thread that sees S_FULL(g) releases it.  V(g) is released by a commit after
  // PV(g); the softmax also waits on that phase to know that PV(g) no longer reads P_b or O.
  static constexpr int K_FULL = 26;    // [6]
  static constexpr int K_EMPTY = 32;   // [6]
  static constexpr int V_READY = 38;   // [6] V landed and, on a boundary tile, zeroed
  static constexpr int V_FULL = 44;    // [6]
  static constexpr int V_EMPTY = 50;   // [6] PV of this stage's tile done
  static constexpr int kMaxStages = 6; // slots 0..55 fit the 512-byte block
  static constexpr int S_FULL = 12;    // [2]
  static constexpr int S_FREE = 14;    // [2] both warpgroups have read S_b out
  static constexpr int P_FULL = 16;    // [2] both warpgroups have written P_b
  static constexpr int Q_FULL = 19;
  static constexpr int Q_EMPTY = 20;
  static constexpr int DRAIN = 21;
};
// named barrier of the two softmax warpgroups (id 0 is __syncthreads)
constexpr int kSoftBar = 1;

// Packed two-lane fp32 arithmetic and three-input max: the softmax warps share their
// schedulers with the MMA-issuing warp, so every instruction they save is issue time the
// tensor pipe's feeder gets back.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float m;
  asm("max.f32 %0, %1, %2, %3;\n" : "=f"(m) : "f"(a), "f"(b), "f"(c));
  return m;
}
// (y0, y1) = (x0, x1) * a + c
__device__ __forceinline__ void fma2f(float& y0, float& y1, float x0, float x1, float a, float c) {
  asm("{\n .reg .b64 x, a, c, y;\n mov.b64 x, {%2, %3};\n mov.b64 a, {%4, %4};\n"
      " mov.b64 c, {%5, %5};\n fma.rn.f32x2 y, x, a, c;\n mov.b64 {%0, %1}, y;\n}\n"
      : "=f"(y0), "=f"(y1)
      : "f"(x0), "f"(x1), "f"(a), "f"(c));
}
// (s0, s1) += (x0, x1)
__device__ __forceinline__ void add2f(float& s0, float& s1, float x0, float x1) {
  asm("{\n .reg .b64 s, x;\n mov.b64 s, {%0, %1};\n mov.b64 x, {%2, %3};\n"
      " add.rn.f32x2 s, s, x;\n mov.b64 {%0, %1}, s;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(x0), "f"(x1));
}

struct PfPiece {
  UnitRec ur;
  SegRec sg;
  KeyTiles kt;
  int64_t ta, tb;
  int slot;
};

template <int BN>
__device__ __forceinline__ bool pf_next(PieceWalk& w, PfPiece& pc, int64_t rows) {
  if (!walk_next(w, pc.ur, pc.ta, pc.tb)) return false;
  pc.kt = key_tiles(pc.ur.lo, pc.ur.hi, rows, BN);
  // the unit record carries its segment's entry and mode: no second dependent load
  pc.sg.q_start = pc.ur.q_start;
  pc.sg.q_len = pc.ur.q_len;
  pc.sg.col = pc.ur.col;
  pc.sg.kv_end = pc.ur.kv_end;
  pc.sg.causal = pc.ur.causal;
  pc.sg.window = pc.ur.window;
  pc.slot = (int)(blockIdx.x - pc.ur.g_first);
  return true;
}

template <int D>
__global__ void __launch_bounds__(PfCfg<D>::THREADS, 1)
    sdpa_prefill_kernel(const AttnArgs A, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  using C = PfCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  griddep_wait();    // the scheduler's output
  griddep_launch();
  {
    // no tiles for this CTA in any phase (or none on the route): the whole CTA leaves
    // before any setup, after one round of header loads
    PieceWalk probe;
    walk_begin(probe, A.ws, kRoutePrefill);
    if (!walk_phase(probe)) return;
  }

  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V,
                 sBar = sbase + C::OFF_BAR;
  auto bar = [&](int i) { return sBar + 8u * (uint32_t)i; };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int W_PROD_K = C::SOFT_WARPS, W_PROD_V = C::SOFT_WARPS + 1, W_MMA = C::SOFT_WARPS + 2;
  volatile int* abort = &s_abort;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(PfBars::K_FULL + s), 1);
      mbar_init(bar(PfBars::K_EMPTY + s), 1);
      mbar_init(bar(PfBars::V_FULL + s), 1);
      mbar_init(bar(PfBars::V_EMPTY + s), 1);
      mbar_init(bar(PfBars::V_READY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(PfBars::S_FULL + b), 1);
      mbar_init(bar(PfBars::S_FREE + b), 32 * C::SOFT_WARPS);
      mbar_init(bar(PfBars::P_FULL + b), 32 * C::SOFT_WARPS);
    }
    mbar_init(bar(PfBars::Q_FULL), 1);
    mbar_init(bar(PfBars::Q_EMPTY), 1);
    mbar_init(bar(PfBars::DRAIN), 1);
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
    // One warp streams Q and K tiles, the other V tiles: K(g) is released as soon as S(g)
    // completes, so the K warp can run ahead while the V warp waits for PV to free V slots.
    const bool is_k = warp == W_PROD_K;
    PieceWalk wk;
    walk_begin(wk, A.ws, kRoutePrefill);
    PfPiece pc;
    uint32_t gt = 0, pi = 0;  // tiles and pieces whose copies this warp started
    bool ok = true;
    while (ok && pf_next<C::BN>(wk, pc, A.rows)) {
      const int hk = pc.ur.hk;
      if (is_k && lane == 0) {
        ok = mbar_wait(bar(PfBars::Q_EMPTY), (pi & 1) ^ 1, abort);
        if (ok) {
          mbar_expect_tx(bar(PfBars::Q_FULL), C::Q_BYTES);
          const int qrow = pc.sg.q_start + (int)(((int64_t)pc.ur.rb * C::BM) / A.group);
#pragma unroll
          for (int c = 0; c < C::NREG; ++c)
            tma_load_3d(sQ + c * (C::BM * 128), &tmQ, bar(PfBars::Q_FULL), 64 * c, hk * A.group, qrow);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (is_k) ++pi;
      const int n = (int)(pc.tb - pc.ta);
      for (int j = 0; ok && j < n; ++j, ++gt) {
        const int s = gt % C::STAGES;
        const uint32_t use = gt / C::STAGES;
        int64_t j0;
        int valid;
        key_tile(pc.kt, pc.ta + j, C::BN, &j0, &valid);
        const int row0 = (int)(j0 % A.rows);
        if (is_k) {
          if (lane == 0) {
            ok = mbar_wait(bar(PfBars::K_EMPTY + s), (use & 1) ^ 1, abort);
            if (ok) {
              mbar_expect_tx(bar(PfBars::K_FULL + s), C::KV_BYTES);
#pragma unroll
              for (int c = 0; c < C::NREG; ++c)
                tma_load_4d(sK + s * C::KV_BYTES + c * (C::BN * 128), &tmK, bar(PfBars::K_FULL + s),
                            64 * c, hk, pc.sg.col, row0);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;  // this tile's copy was not started
          continue;
        }
        if (lane == 0) {
          ok = mbar_wait(bar(PfBars::V_EMPTY + s), (use & 1) ^ 1, abort);
          if (ok) {
            // a full tile needs no zeroing: V_READY goes ahead of the copy, so it is complete
            // whenever V_FULL is
            if (valid == C::BN) mbar_arrive(bar(PfBars::V_READY + s));
            mbar_expect_tx(bar(PfBars::V_FULL + s), C::KV_BYTES);
#pragma unroll
            for (int c = 0; c < C::NREG; ++c)
              tma_load_4d(sV + s * C::KV_BYTES + c * (C::BN * 128), &tmV, bar(PfBars::V_FULL + s),
                          64 * c, hk, pc.sg.col, row0);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (valid < C::BN) {
          // V rows past the last visible key: wait for the tile, then zero them
          ok = mbar_wait(bar(PfBars::V_FULL + s), use & 1, abort);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            ++gt;  // its copy was started
            break;
          }
          const int bytes = (C::BN - valid) * 128;
#pragma unroll
          for (int c = 0; c < C::NREG; ++c) {
            uint8_t* reg = smem + C::OFF_V + s * C::KV_BYTES + c * (C::BN * 128) + valid * 128;
            for (int o = lane * 16; o < bytes; o += 32 * 16)
              *reinterpret_cast<uint4*>(reg + o) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(PfBars::V_READY + s));
        }
      }
    }
    // drain: the copies this warp started must land before the CTA can exit (immediate on
    // the normal path, where the MMA warp already consumed every stage and Q tile); each
    // wait is bounded on its own
    if (lane == 0) {
      const uint32_t first = gt > (uint32_t)C::STAGES ? gt - C::STAGES : 0u;
      for (uint32_t g = first; g < gt; ++g) {
        int own = 0;
        mbar_wait(bar((is_k ? PfBars::K_FULL : PfBars::V_FULL) + g % C::STAGES), (g / C::STAGES) & 1, &own);
      }
      if (is_k && pi > 0) {
        int own = 0;
        mbar_wait(bar(PfBars::Q_FULL), (pi - 1) & 1, &own);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop with warp-uniform values; one elected lane issues
    // each MMA and commit.
    {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, C::BN, false, false);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, false, true);
      PieceWalk wk;
      walk_begin(wk, A.ws, kRoutePrefill);
      PfPiece pc;
      uint32_t gt = 0, pi = 0;
      bool ok = true;
      // Descriptors differ only in their start-address field (bits 0-13, address / 16), so
      // each MMA's operands are a base descriptor plus a byte offset / 16.
      const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);
      const uint64_t k_desc = sdesc_sw128(sK, 16, 1024);
      const uint64_t v_desc = sdesc_sw128(sV, C::BN * 128, 1024);
      // Issue order S(0) S(1) | S(2) PV(0) | S(3) PV(1) | ...: S(g+2) goes out as soon as
      // the softmax has read S(g) out of S_b (S_FREE), PV(g) once P(g) is in P_b (P_FULL),
      // so the tensor pipe computes the next scores while the softmax works on this tile.
      // The MMA queue is shallow: a blocking wait here leaves the pipe idle for its
      // latency.  So the next waits are tested (non-blocking) between the last MMAs of a
      // block, where the test's latency hides behind MMA issue, and the blocking waits run
      // only when a test came back negative.
      constexpr int KS = D / 16, KP = C::BN / 16;  // k-steps of S and of PV
      auto s_deps = [&](uint32_t g) -> bool {
        return __all_sync(0xffffffffu,
                          mbar_wait(bar(PfBars::K_FULL + g % C::STAGES), (g / C::STAGES) & 1, abort) &&
                              mbar_wait(bar(PfBars::S_FREE + (g & 1)), ((g >> 1) & 1) ^ 1, abort));
      };
      // (the tests' results are voted on only after the block, so no MMA waits for them)
      auto s_test = [&](uint32_t g) -> bool {
        return mbar_test_wait(bar(PfBars::K_FULL + g % C::STAGES), (g / C::STAGES) & 1) &
               mbar_test_wait(bar(PfBars::S_FREE + (g & 1)), ((g >> 1) & 1) ^ 1);
      };
      auto pv_test = [&](uint32_t g) -> bool {
        return mbar_test_wait(bar(PfBars::P_FULL + (g & 1)), (g >> 1) & 1) &
               mbar_test_wait(bar(PfBars::V_FULL + g % C::STAGES), (g / C::STAGES) & 1);
      };
      // S(g) = Q K(g)^T into S_b; tests PV(tg)'s barriers on the way when `test`
      auto issue_s = [&](uint32_t g, bool test, uint32_t tg) -> bool {
        const int s = g % C::STAGES, b = g & 1;
        const uint64_t kd = k_desc + (uint64_t)((s * C::KV_BYTES) >> 4);
        const uint32_t d = tmem + C::S_COL0 + b * C::BN;
        bool pre = false;
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          if (k == KS - 2 && test) pre = pv_test(tg);
          const uint32_t off = ((k >> 2) * (C::BM * 128) + (k & 3) * 32) >> 4;
          const uint32_t offk = ((k >> 2) * (C::BN * 128) + (k & 3) * 32) >> 4;
          tc_mma_ss_w(d, q_desc + off, kd + offk, IDESC_QK, k > 0 ? 1u : 0u);
        }
        tc_commit_w(bar(PfBars::S_FULL + b));
        return test && __all_sync(0xffffffffu, pre);
      };
      // O (+)= P(g) V(g), A = P_b from tensor memory; tests S(tg)'s barriers when `test`
      auto issue_pv = [&](uint32_t g, uint32_t acc0, bool test, uint32_t tg) -> bool {
        const int s = g % C::STAGES, b = g & 1;
        const uint64_t vd = v_desc + (uint64_t)((s * C::KV_BYTES) >> 4);
        const uint32_t pa = tmem + C::P_COL + b * (C::BN / 2), od = tmem + C::O_COL;
        bool pre = false;
#pragma unroll
        for (int k = 0; k < KP; ++k) {
          if (k == KP - 2 && test) pre = s_test(tg);
          tc_mma_ts_w(od, pa + 8 * k, vd + (uint64_t)((k * 16 * 128) >> 4), IDESC_PV, k > 0 ? 1u : acc0);
        }
        tc_commit_w(bar(PfBars::V_EMPTY + s));  // V(g) free, and PV(g) done with P_b and O
        return test && __all_sync(0xffffffffu, pre);
      };
      while (ok && pf_next<C::BN>(wk, pc, A.rows)) {
        const int n = (int)(pc.tb - pc.ta);
        ok = __all_sync(0xffffffffu, mbar_wait(bar(PfBars::Q_FULL), pi & 1, abort)) && s_deps(gt) &&
             (n < 2 || s_deps(gt + 1));
        if (!ok) break;
        tc_fence_after();
        issue_s(gt, false, 0);
        if (n > 1) issue_s(gt + 1, false, 0);
        if (n <= 2) tc_commit_w(bar(PfBars::Q_EMPTY));  // every S of this piece has been issued
        bool pre_s = false;  // S(g+2)'s barriers were seen complete by the tests
        for (int j = 0; j < n; ++j) {
          const uint32_t g = gt + j;
          const int b = g & 1, s = g % C::STAGES;
          // V_READY is awaited on short tiles only (the V producer zeroes the rest of such a
          // tile): the producer arrives on it for every tile (before the copy, or after
          // zeroing the rows past the last key), so at this wait the barrier has completed
          // exactly the phases of earlier uses and this one.
          int64_t tj0;
          int tvalid;
          key_tile(pc.kt, pc.ta + j, C::BN, &tj0, &tvalid);
          const bool tail = tvalid < C::BN;
          bool pre_pv = false;
          if (j + 2 < n) {
            if (!pre_s) {
              ok = s_deps(g + 2);
              if (!ok) break;
            }
            tc_fence_after();
            pre_pv = issue_s(g + 2, !tail, g);
            if (j + 3 == n) tc_commit_w(bar(PfBars::Q_EMPTY));
          }
          if (!pre_pv) {
            ok = __all_sync(0xffffffffu,
                            mbar_wait(bar(PfBars::P_FULL + b), (g >> 1) & 1, abort) &&
                                mbar_wait(bar(PfBars::V_FULL + s), (g / C::STAGES) & 1, abort) &&
                                (!tail || mbar_wait(bar(PfBars::V_READY + s), (g / C::STAGES) & 1, abort)));
            if (!ok) break;
          }
          tc_fence_after();
          pre_s = issue_pv(g, j > 0 ? 1u : 0u, j + 3 < n, g + 3);
        }
        gt += n;
        ++pi;
      }
      // drain: wait (bounded) until every MMA this thread issued has finished
      tc_commit_w(bar(PfBars::DRAIN));
      int dummy = 0;
      mbar_wait(bar(PfBars::DRAIN), 0, &dummy);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    // Both warpgroups work on every tile: warpgroup wg takes key columns
    // [wg*HALF, (wg+1)*HALF) of S_b, thread = row = tensor-memory lane.  They share one
    // running max per row, keep their own partial row sums, and rescale / finalise their
    // own half of O's columns.  Values are swapped through tensor memory (same lane = same
    // row): each warpgroup writes into a column of the OTHER's half of P_b, which only that
    // other warpgroup reads and later overwrites with its P, so no slot is overwritten
    // before its reader is done.  The named barrier that
    // carries the max exchange also ANDs the CTA's abort state, so the two warpgroups
    // always leave together; waits between two such barriers record a failure instead of
    // leaving at once.
    const int wg = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_off + C::S_COL0 + wg * C::HALF;
    const uint32_t t_p = tmem + lane_off + C::P_COL + wg * (C::HALF / 2);
    const uint32_t t_o = tmem + lane_off + C::O_COL + wg * (D / 2);
    const uint32_t t_xw = tmem + lane_off + C::P_COL + (wg == 0 ? C::HALF / 2 : 0);
    const uint32_t t_xr = tmem + lane_off + C::P_COL + (wg == 0 ? 0 : C::HALF / 2);
    const float sl2 = A.scale_log2;
    // PV(g) finished (its commit completes stage g % STAGES's V_EMPTY phase)
    auto pv_done = [&](uint32_t g) -> bool {
      return mbar_wait(bar(PfBars::V_EMPTY + g % C::STAGES), (g / C::STAGES) & 1, abort);
    };
    PieceWalk wk;
    walk_begin(wk, A.ws, kRoutePrefill);
    PfPiece pc;
    uint32_t gt = 0;
    bool ok = true;
    while (ok && pf_next<C::BN>(wk, pc, A.rows)) {
      const UnitRec& ur = pc.ur;
      const SegRec& sg = pc.sg;
      const bool live = row < ur.rows;
      const int64_t r = (int64_t)ur.rb * C::BM + row;
      const int qi = (int)(r / A.group);
      int64_t rlo = 1, rhi = 0;  // padding rows see nothing
      if (live) {
        const RowWin w = row_window(qi, sg.q_len, sg.kv_end, sg.causal, sg.window);
        rlo = w.lo;
        rhi = w.hi;
      }
      const int n = (int)(pc.tb - pc.ta);
      float m_use = -INFINITY, l = 0.f;
      bool okp = true;  // no wait failed since the last barrier
      for (int j = 0; j < n; ++j) {
        const uint32_t g = gt + j;
        const int b = g & 1;
        const bool okw = mbar_wait(bar(PfBars::S_FULL + b), (g >> 1) & 1, abort);
        // P_b was last read by PV(g-2): tested here, its answer used after the max
        const uint32_t g2 = g - 2;
        const bool pv2 = g < 2 || mbar_test_wait(bar(PfBars::V_EMPTY + g2 % C::STAGES), (g2 / C::STAGES) & 1);
        // this half's visible columns of the tile (its keys [tj0, tj0 + tvalid) exist)
        int64_t tj0;
        int tvalid;
        key_tile(pc.kt, pc.ta + j, C::BN, &tj0, &tvalid);
        const int64_t j0 = tj0 + wg * C::HALF;
        const int64_t hv = min(max((int64_t)tvalid - wg * C::HALF, (int64_t)0), (int64_t)C::HALF);
        const int vlo = okw ? (int)min(max(rlo - j0, (int64_t)0), hv) : 0;
        const int vhi = okw ? (int)min(max(rhi - j0, (int64_t)0), hv) : 0;
        float x[C::HALF];
        if (okw) {
          tc_fence_after();
          if constexpr (C::HALF == 64)
            tmem_ld64(t_s + b * C::BN, x);
          else
            tmem_ld32(t_s + b * C::BN, x);
        }
        tc_fence_before();
        mbar_arrive(bar(PfBars::S_FREE + b));
        if (threadIdx.x == 0 && okw) mbar_arrive(bar(PfBars::K_EMPTY + g % C::STAGES));  // S(g) done
        // columns outside [vlo, vhi) (masked keys, stale cells past the last key) -> -inf
        if (vlo > 0 || vhi < C::HALF) {
#pragma unroll
          for (int k = 0; k < C::HALF; ++k) x[k] = (k >= vlo && k < vhi) ? x[k] : -INFINITY;
        }
        float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int k = 4; k < C::HALF; k += 2) mx4[(k >> 1) & 3] = max3f(mx4[(k >> 1) & 3], x[k], x[k + 1]);
        // scale is positive, so max(scale * s) = scale * max(s)
        const float mx = fmaxf(max3f(mx4[0], mx4[1], mx4[2]), mx4[3]) * sl2;
        // Fast path: no row of either half has a tile max above m_use + 2^8, so every running
        // max stays as it is and nothing needs exchanging.  The barrier's AND also carries
        // the wait results; a false AND takes the slow path, whose barrier tells them apart.
        const bool calm = mx <= m_use + 8.f;
        const bool fast = bar_and(kSoftBar, 32 * C::SOFT_WARPS, ok && okp && okw && calm);
        if (!fast) {
          if (!__all_sync(0xffffffffu, pv2)) okp = okp && __all_sync(0xffffffffu, pv_done(g2));
          if (okp && okw) {
            tc_fence_after();
            tmem_st1(t_xw + b * (C::BN / 2), mx);
          }
          tc_fence_before();
          ok = bar_and(kSoftBar, 32 * C::SOFT_WARPS, ok && okp && okw);
          if (!ok) break;
          tc_fence_after();
          const float m_tile = fmaxf(mx, tmem_ld1(t_xr + b * (C::BN / 2)));
          const float m_new = fmaxf(m_use, m_tile);
          const bool resc = m_new > m_use + 8.f;  // false while nothing is visible
          const float alpha = resc ? exp2_approx(m_use - m_new) : 1.f;
          const bool need_o = resc && j > 0 && m_use != -INFINITY;
          if (__any_sync(0xffffffffu, need_o)) {
            // rescale this half of O once PV(g-1) has landed in it
            okp = okp && __all_sync(0xffffffffu, pv_done(g - 1));
            if (okp) {
              tc_fence_after();
              const float f = need_o ? alpha : 1.f;
#pragma unroll 1
              for (int c = 0; c < D / 64; ++c) {
                float o[32];
                tmem_ld32(t_o + 32 * c, o);
#pragma unroll
                for (int k = 0; k < 32; ++k) o[k] *= f;
                tmem_st32(t_o + 32 * c, o);
              }
            }
          }
          if (resc) {
            m_use = m_new;
            l *= alpha;
          }
        } else if (!__all_sync(0xffffffffu, pv2)) {
          okp = okp && __all_sync(0xffffffffu, pv_done(g2));
        }
        tc_fence_after();
        const float nmu = m_use == -INFINITY ? 0.f : -m_use;
        // p = 2^(scale*s - m) (masked columns give 0), row sum; P as bf16 pairs into P_b
        float sum8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pw[C::HALF / 2];
#pragma unroll
        for (int k = 0; k < C::HALF / 2; ++k) {
          float a0, a1;
          fma2f(a0, a1, x[2 * k], x[2 * k + 1], sl2, nmu);
          const float p0 = exp2_approx(a0), p1 = exp2_approx(a1);
          add2f(sum8[(2 * k) & 7], sum8[(2 * k + 1) & 7], p0, p1);
          pw[k] = pack_bf16x2(p0, p1);
        }
        if (okp) {
          if constexpr (C::HALF == 64)
            tmem_st32u(t_p + b * (C::BN / 2), pw);
          else
            tmem_st16u(t_p + b * (C::BN / 2), pw);
        }
        l += ((sum8[0] + sum8[1]) + (sum8[2] + sum8[3])) + ((sum8[4] + sum8[5]) + (sum8[6] + sum8[7]));
        tc_fence_before();
        mbar_arrive(bar(PfBars::P_FULL + b));
      }
      if (!ok) break;
      gt += n;
      // epilogue: once the piece's last PV is done, swap the partial row sums through the
      // exchange slots of that PV's (now idle) P buffer - the one the next piece writes
      // second, behind a barrier - then normalise (direct) or write a partial
      const bool okw = pv_done(gt - 1);
      const uint32_t xb = ((gt - 1) & 1) * (C::BN / 2);
      if (okw) {
        tc_fence_after();
        tmem_st1(t_xw + xb, l);
      }
      tc_fence_before();
      ok = bar_and(kSoftBar, 32 * C::SOFT_WARPS, ok && okp && okw);
      if (!ok) break;
      tc_fence_after();
      const float L = l + tmem_ld1(t_xr + xb);
      const bool direct = ur.nslots == 1;
      const int h = ur.hk * A.group + (int)(r % A.group);
      __nv_bfloat16* orow = A.out + ((int64_t)sg.q_start + qi) * A.o_rs + (int64_t)h * A.o_hs + wg * (D / 2);
      const int64_t pidx = ur.slot_base + (int64_t)pc.slot * ur.rows + row;
      float* prow = A.ws.part_o[kRoutePrefill] + pidx * D + wg * (D / 2);
      // a row with no visible key has L = 0 and writes zeros (never 0 * O)
      const bool empty = !(L > 0.f);
      const float w = direct ? 1.f / L : 1.f;
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
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
      if (live && !direct && wg == 0) A.ws.part_ml[kRoutePrefill][pidx] = make_float2(m_use, L);
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

template __global__ void sdpa_prefill_kernel<256>(const AttnArgs, const __grid_constant__ CUtensorMap,
                                                  const __grid_constant__ CUtensorMap,
                                                  const __grid_constant__ CUtensorMap);

// The prefill kernel of a head dim: this one at D = 256, the two-tile kernel otherwise.
const void* prefill_kernel_ptr(int D) {
  return D == 256 ? (const void*)sdpa_prefill_kernel<256> : prefill_pair_kernel_ptr(D);
}
int prefill_smem_bytes(int D) { return D == 256 ? PfCfg<256>::SMEM : prefill_pair_smem_bytes(D); }
int prefill_block_threads(int D) { return D == 256 ? PfCfg<256>::THREADS : prefill_pair_block_threads(D); }
int prefill_tile_keys(int D) { return D == 256 ? PfCfg<256>::BN : kPrefillTile; }

}  // namespace sdpa
