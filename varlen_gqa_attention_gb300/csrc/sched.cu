// sched.cu - device-side segment scheduler.
//
// Walks the segment table on the device ("[executorch][cuda] Add a length-aware Triton SDPA
// over per-sequence KV columns", PR description: lengths are read on device, so one captured
// graph serves any mix of sequence lengths) and turns it into work for the attention kernels:
//   1. validates each segment (SDPA_SEG_* bits);
//   2. claims packed rows for valid segments, dropping every segment that shares a row with
//      another one (SDPA_SEG_OVERLAP);
//   3. routes each remaining segment to the split-K or the tensor-memory prefill kernel and
//      cuts it into units (segment, KV head, block of packed (query row, head) rows);
//   4. counts each unit's key tiles over the union of its rows' visible intervals and lays
//      all units' tiles end to end on a line of cost units (tile_cost: 4 or 6 per split-K
//      tile by its unit's rows, 1 per prefill tile), each unit's behind lead placeholders
//      for the cost of starting a piece (lead_cost); the line is cut into at most four phases whose
//      re-read K/V fits the L2 budget; within a phase CTA g of G owns the tiles whose start
//      lies in [g*W/G, (g+1)*W/G) (a stream-K split, so every CTA gets the same cost whatever
//      the length mix; G is capped at W over the costliest tile, so that every CTA owns a
//      tile of each unit its share crosses), the CTAs whose share starts in a unit are
//      recorded against it, and each (unit, CTA) pair gets a slot of partial results unless
//      the unit has a single CTA, which then writes `out` itself;
//   5. publishes the records, a per-row record for the combine pass and a flag that tells
//      the combine pass whether it has any work.
// One CTA of 512 threads does all of it.  The work is small and serial (a chain of dependent
// steps with a barrier between each), so the cost of a call is the length of that chain, not
// its arithmetic; two shorter chains cover the usual decode and mixed steps:
//   * at most 32 segments (and 8192 packed rows): steps 1-3 run in warp 0, one segment per
//     lane, with shuffles (pairwise overlap test, unit-base scan) and no barrier, while the
//     other warps clear the row owner map;
//   * at most 512 units: one unit per thread, its record kept in registers; one-barrier scans,
//     and each thread writes the phase bases that start at the next unit from its own prefix.
// Otherwise block-wide steps over contiguous ranges per thread.  Segment tables of up to 1024
// segments, up to 8192 packed rows and up to 1024 units are built in shared memory; larger
// calls run the same steps on the workspace copies.
#include "common.cuh"

namespace sdpa {


// Exclusive block scan of N int64 values per thread (N <= warps): v becomes this thread's
// prefix, tot the block totals.  Warp k scans the warp totals of value k, so the N scans
// cost the barriers of one.
template <int N>
__device__ void block_scan(int64_t (&v)[N], int64_t (&tot)[N], int64_t* sh /*[N * 32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int64_t x[N];
#pragma unroll
  for (int k = 0; k < N; ++k) {
    x[k] = v[k];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x[k], o);
      if (lane >= o) x[k] += y;
    }
    if (lane == 31) sh[k * 32 + warp] = x[k];
  }
  __syncthreads();
  if (warp < N) {
    int64_t w = lane < nw ? sh[warp * 32 + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) sh[warp * 32 + lane] = w;  // inclusive warp totals
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < N; ++k) {
    const int64_t base = warp > 0 ? sh[k * 32 + warp - 1] : 0;
    tot[k] = sh[k * 32 + nw - 1];
    v[k] = base + x[k] - v[k];
  }
  __syncthreads();
}

// Exclusive scan of N int64 values per thread over one route's threads, with one barrier.
// The threads of a route are whole warps (route r of warp w: wroute(w), 0 for none); warps of
// no route skip the shuffles (a shuffle takes the SM's shuffle unit for a cycle, whichever
// warp issues it, so idle warps would slow the others).  tot: the route's totals.
template <int N, typename F>
__device__ void route_scan(int64_t (&v)[N], int64_t (&tot)[N], int64_t* sh /*[N * 32]*/, F wroute) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int r = wroute(warp);
  int64_t x[N];
  if (r != 0) {
#pragma unroll
    for (int k = 0; k < N; ++k) {
      x[k] = v[k];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x[k], o);
        if (lane >= o) x[k] += y;
      }
      if (lane == 31) sh[k * 32 + warp] = x[k];
    }
  }
  __syncthreads();
  if (r == 0) return;
  const bool mine = lane < nw && wroute(lane) == r;
#pragma unroll
  for (int k = 0; k < N; ++k) {
    int64_t w = mine ? sh[k * 32 + lane] : 0;
    for (int o = 1; o < nw; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    const int64_t base = __shfl_sync(0xffffffffu, w, warp > 0 ? warp - 1 : 0);
    tot[k] = __shfl_sync(0xffffffffu, w, nw - 1);
    v[k] = (warp > 0 ? base : 0) + x[k] - v[k];
  }
}

// Phase of a unit whose route's earlier units re-read `bytes` of K/V: bytes / kPhaseBytes,
// capped (kPhaseBytes = 3 * 2^24, so a shift and a 32-bit division by 3).
static_assert(kPhaseBytes == (3ll << 24), "phase budget");
__device__ __forceinline__ int phase_of(int64_t bytes, int cap) {
  const uint64_t m = (uint64_t)bytes >> 24;
  return m >= 3ull * (uint64_t)cap ? cap : (int)((uint32_t)m / 3u);
}

// Sum of one float per thread, the same value (same order) in every thread; one barrier.
// sh: 32 floats used by this call only.
__device__ float block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  float t = 0.f;
  for (int w = 0; w < nw; ++w) t += sh[w];
  return t;
}

// Contiguous range of n items owned by this thread.
__device__ __forceinline__ void my_range(int64_t n, int64_t* a, int64_t* b) {
  const int64_t per = udiv(n + blockDim.x - 1, blockDim.x);
  *a = min(n, per * threadIdx.x);
  *b = min(n, *a + per);
}

__device__ __forceinline__ void load_seg(const SchedArgs& A, int s, int32_t* seg) {
  if (A.use_inline) {
    seg[0] = A.inl[0]; seg[1] = A.inl[1]; seg[2] = A.inl[2]; seg[3] = A.inl[3];
  } else {
    int4 v = reinterpret_cast<const int4*>(A.seq_info)[s];
    seg[0] = v.x; seg[1] = v.y; seg[2] = v.z; seg[3] = v.w;
  }
}

__device__ __forceinline__ int rows_per_unit(const SchedArgs& A, int route) {
  return route == kRoutePrefill ? prefill_unit_rows(A.D) : kSplitkRows;
}
__device__ __forceinline__ int tile_len(const SchedArgs& A, int route) {
  return route == kRoutePrefill ? A.tile_pf : kSplitkTile;
}

// Route of a live segment.  The prefill kernel takes segments that fill at least one
// 128-row tile (on a ring store too: its key tiles stop at the wrap, so a TMA box never
// wraps), when the call holds enough such work to pay for that kernel's fixed cost (`big`:
// the segments' prefill_work sums to at least kPrefillMinWork); everything else, and
// everything when the prefill kernel is unusable, goes to the split-K kernel.
__device__ __forceinline__ int route_of(const SchedArgs& A, int32_t q_len, bool big) {
  const int64_t R = (int64_t)q_len * A.group;
  if (A.policy == SDPA_ROUTE_SPLITK || !A.prefill_ok) return kRouteSplitk;
  if (A.policy == SDPA_ROUTE_PREFILL) return kRoutePrefill;
  return R >= kPrefillRows && big ? kRoutePrefill : kRouteSplitk;
}
// A live segment's share of the prefill route's work measure: packed rows * needed key
// span * Hkv * D when it fills a 128-row tile, else 0 (in fp32: no overflow, ample for a
// threshold, and fast; fp64 runs at a small fraction of the fp32 rate here).
__device__ __forceinline__ float prefill_work(const SchedArgs& A, int32_t q_len, int32_t kv_end, int32_t window) {
  const int64_t R = (int64_t)q_len * A.group;
  if (R < kPrefillRows) return 0.f;
  int64_t span = kv_end;
  if (window > 0) span = min(span, (int64_t)q_len + window - 1);
  return (float)R * (float)span * (float)A.Hkv * (float)A.D;
}

// A segment's entry as the unit builder reads it.
struct SegView {
  int32_t q_start, q_len, col, kv_end, nrb, ubase, causal, window;
};

// Record of unit uq of route q, which belongs to segment s: its (KV head, row block), rows,
// key range and key tiles.  *span: the unit's length on its route's tile line (the lead
// placeholders and its key tiles; 0 when no key is visible); *reuse: the K/V bytes its
// (segment, KV head) group reads again, counted once, on the group's last unit, and only for
// groups of several units (phases are cut on these).
__device__ __forceinline__ UnitRec make_unit(const SchedArgs& A, int s, const SegView& g, int q, int64_t uq,
                                             int64_t* span, int64_t* reuse) {
  const int rpu = rows_per_unit(A, q), tl = tile_len(A, q);
  UnitRec ur;
  const int64_t j = uq - g.ubase;
  const int64_t jh = udiv(j, g.nrb);
  ur.seg = s;
  ur.q_start = g.q_start;
  ur.q_len = g.q_len;
  ur.col = g.col;
  ur.kv_end = g.kv_end;
  ur.causal = g.causal;
  ur.window = g.window;
  ur.hk = (int32_t)jh;
  ur.rb = (int32_t)(j - jh * g.nrb);
  const int64_t R = (int64_t)g.q_len * A.group;
  const int64_t r0 = (int64_t)ur.rb * rpu;
  ur.rows = (int32_t)min((int64_t)rpu, R - r0);
  const int i0 = (int)udiv(r0, A.group), i1 = (int)udiv(r0 + ur.rows - 1, A.group);
  const RowWin w0 = row_window(i0, g.q_len, g.kv_end, g.causal, g.window);
  const RowWin w1 = row_window(i1, g.q_len, g.kv_end, g.causal, g.window);
  ur.lo = w0.lo;  // lo and hi grow with the query row
  ur.hi = max(w1.hi, w0.lo);
  // key tiles: the prefill kernel's stop at a ring wrap (two TMA ranges), the split-K
  // kernel's wrap per row
  const int64_t nt = q == kRoutePrefill ? key_tiles(ur.lo, ur.hi, A.rows, tl).n
                                        : (ur.hi > ur.lo ? udiv((int64_t)(ur.hi - ur.lo) + tl - 1, tl) : 0);
  ur.nslots = 0;
  ur.g_first = 0;
  ur.ntiles = (int32_t)nt;
  ur.phase = 0;
  ur.tile_base = 0;
  ur.slot_base = 0;
  *span = nt > 0 ? nt * tile_cost(q, ur.rows) + lead_cost(q) : 0;
  *reuse = 0;
  if (g.nrb >= 2 && ur.rb == g.nrb - 1) {
    int64_t sp = g.kv_end;
    if (g.window > 0) sp = min(sp, (int64_t)g.q_len + g.window - 1);
    *reuse = sp * (int64_t)A.D * 4;
  }
  return ur;
}

// Stream-K placement of a unit whose tile_base and phase are set, within its phase: CTA g of
// G_p = min(G, W_p) owns [g W_p / G_p, (g+1) W_p / G_p); G_p <= W_p makes every working CTA
// own a tile, so the owners of a unit's tiles are consecutive CTAs that all work on it
// (nslots is exact).  Records the CTAs whose share starts inside the unit's span in the
// per-CTA start table.  pb: the route's phase bases.  Returns the unit's partial rows (its
// slots, when several CTAs share it).
// Whether phase p of route q takes one whole unit per CTA: its units (pu0[p], pu0[p+1]) are
// at most the CTAs, and the longest (pmax, in line units) costs no more than an even
// stream-K share of the phase (W_p / G) plus what cutting units costs: partial slots written
// by the attention kernel and merged by the combine pass, about 12 prefill tiles (~8 us) on the
// prefill route and 8 units (2 small tiles) on the split-K route, whose merges overlap its
// tail.  Short, even units (a windowed prefill of many row blocks) then avoid the merges;
// long ones (a 131072-key prefill) keep the stream-K split, which leaves no CTA idle.
__device__ __forceinline__ bool phase_is_aligned(const int64_t* pb, const int64_t* pu0, const int32_t* pmax,
                                                 int p, int64_t G, int q) {
  const int64_t Up = pu0[p + 1] - pu0[p], Wp = pb[p + 1] - pb[p];
  const int64_t M = q == kRouteSplitk ? 8 : 12;
  return Up > 0 && Up <= G && (int64_t)pmax[p] * G <= Wp + M * G;
}

__device__ __forceinline__ int64_t place_unit(const SchedArgs& A, UnitRec& ur, int q, int64_t uq,
                                              const int64_t* pb, const int64_t* pu0, bool aligned) {
  const int64_t nt = ur.ntiles;
  if (nt <= 0) return 0;
  const int64_t G = A.grid[q];
  if (aligned) {  // CTA g of the phase takes its unit g whole and writes `out` itself
    const int64_t g = uq - pu0[ur.phase];
    ur.g_first = (int32_t)g;
    ur.nslots = 1;
    A.ws.first_unit[q][ur.phase * G + g] = (int32_t)uq;
    return 0;
  }
  const int64_t tw = tile_cost(q, ur.rows);
  const int64_t b0 = pb[ur.phase];
  const int64_t Wp = pb[ur.phase + 1] - b0;
  const int64_t Gp = phase_ctas(G, Wp, q);
  const int64_t k0 = ur.tile_base + lead_cost(q) - b0;  // the key tiles, phase-relative
  const int64_t g0 = sk_owner(k0, Wp, Gp);
  const int64_t g1 = sk_owner(k0 + (nt - 1) * tw, Wp, Gp);  // the owners of the first and last tile starts
  ur.g_first = (int32_t)g0;
  ur.nslots = (int32_t)(g1 - g0 + 1);
  // the CTAs whose share starts inside the unit's span: after the owner of the position
  // before the span, up to the owner of its last position
  const int64_t s0 = ur.tile_base - b0, s1 = k0 + nt * tw;
  const int64_t c0 = s0 > 0 ? sk_owner(s0 - 1, Wp, Gp) + 1 : 0;
  const int64_t c1 = sk_owner(s1 - 1, Wp, Gp);
  for (int64_t c = c0; c <= c1; ++c) A.ws.first_unit[q][ur.phase * G + c] = (int32_t)uq;
  return ur.nslots > 1 ? (int64_t)ur.nslots * ur.rows : 0;
}

// Shared-memory staging: segment tables of up to kSegCache rows, the row-owner map of up
// to kRowCache packed rows and up to kUnitCache units (both routes) are built in shared
// memory, so the walk is a chain of block-wide steps with no global round trips, and the
// records are written out once at the end.  Larger calls keep the same steps on the
// workspace copies in global memory.
constexpr int kSegCache = 1024;
constexpr int kRowCache = 8192;
constexpr int kUnitCache = 1024;
constexpr size_t kSchedSmem = (size_t)kSegCache * (16 + 8 + 8 + 8 + 4 + 4) + (size_t)kRowCache * 4 +
                              (size_t)kUnitCache * sizeof(UnitRec);

__global__ void __launch_bounds__(kSchedThreads) sdpa_sched_kernel(SchedArgs A) {
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int64_t sh[4 * 32];
  __shared__ float s_fsum[32];
  __shared__ int64_t s_pb[3][kMaxPhases + 1];
  __shared__ int64_t s_pu0[3][kMaxPhases + 1];  // first unit of each phase; [np] = units
  __shared__ int32_t s_pmax[3][kMaxPhases];      // longest unit span of each phase
  __shared__ int64_t s_U[3], s_np[3];
  __shared__ int32_t s_status, s_work;
  int4* c_seg = reinterpret_cast<int4*>(smem);      // (q_start, q_len, col, kv_end)
  int2* c_mode = reinterpret_cast<int2*>(c_seg + kSegCache);  // (causal, window)
  int2* c_rn = c_mode + kSegCache;                  // (route, nrb)
  int2* c_ub = c_rn + kSegCache;                    // unit bases on routes 1 and 2
  int32_t* c_bits = reinterpret_cast<int32_t*>(c_ub + kSegCache);
  int32_t* c_flag = c_bits + kSegCache;             // overlap flags
  int32_t* c_row = c_flag + kSegCache;              // packed row -> owning segment
  UnitRec* c_unit = reinterpret_cast<UnitRec*>(c_row + kRowCache);

  const Workspace& W = A.ws;
  const int S = A.S;
  const int64_t T = A.T;
  const bool cached = S <= kSegCache;
  const bool rows_cached = cached && T <= kRowCache;
  int32_t* row_map = rows_cached ? c_row : W.row_seg;
  int32_t* flag = cached ? c_flag : W.seg_flag;
  auto seg_of = [&](int s) -> int4 {
    if (cached) return c_seg[s];
    const SegRec r = W.segs[s];
    return make_int4(r.q_start, r.q_len, r.col, r.kv_end);
  };
  auto bits_of = [&](int s) -> int32_t { return cached ? c_bits[s] : W.segs[s].bits; };

  {
    griddep_launch();  // the attention kernels may start launching; they wait for this grid
    if (threadIdx.x == 0) {
      s_status = 0;
      s_work = 0;
    }
    if (threadIdx.x < 3 * kMaxPhases) (&s_pmax[0][0])[threadIdx.x] = 0;
    __syncthreads();

    // 1. validate; clear overlap flags and the row owner map
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
      int32_t g[4];
      load_seg(A, s, g);
      int2 md = make_int2(A.causal, A.window);
      if (A.seg_mode) {
        md = reinterpret_cast<const int2*>(A.seg_mode)[s];
        md.x = md.x != 0;
      }
      const int32_t bits = segment_bits(g[0], g[1], g[2], g[3], T, A.rows, A.cols, md.y);
      if (cached) {
        c_seg[s] = make_int4(g[0], g[1], g[2], g[3]);
        c_bits[s] = bits;
        c_mode[s] = md;
      } else {
        SegRec r;
        r.q_start = g[0]; r.q_len = g[1]; r.col = g[2]; r.kv_end = g[3];
        r.route = kRouteNone; r.nrb = 0; r.bits = bits; r.pad = 0;
        r.ubase[0] = r.ubase[1] = r.ubase[2] = r.ubase[3] = 0;
        r.causal = md.x; r.window = md.y;
        r.pad2[0] = r.pad2[1] = 0;
        W.segs[s] = r;
      }
      flag[s] = 0;
      if (bits) atomicOr(&s_status, bits);
    }
    for (int64_t t = threadIdx.x; t < T; t += blockDim.x) row_map[t] = -1;
    __syncthreads();

    // 2. claim rows; a segment that meets another one marks both.  Teams of threads take
    // segments round-robin: the whole block per segment when segments are few, one warp per
    // segment when there are at least as many segments as warps.
    {
      int team = blockDim.x;
      while (team > 32 && team * S > (int)blockDim.x * 2) team >>= 1;
      const int nteam = blockDim.x / team, tm = threadIdx.x / team, ti = threadIdx.x % team;
      for (int s = tm; s < S; s += nteam) {
        if (bits_of(s)) continue;
        const int4 g = seg_of(s);
        for (int i = ti; i < g.y; i += team) {
          const int old = atomicCAS(&row_map[g.x + i], -1, s);
          if (old != -1) {
            atomicExch(&flag[s], 1);
            atomicExch(&flag[old], 1);
          }
        }
      }
    }
    __syncthreads();

    // 3. route each live segment and count its units (contiguous segment ranges per thread);
    // first the call's prefill work, which decides whether the prefill route is taken
    int64_t sa, sb;
    my_range(S, &sa, &sb);
    float pw = 0.f;
    for (int64_t s = sa; s < sb; ++s) {
      const int4 g = seg_of((int)s);
      if (bits_of((int)s) == 0 && !flag[s] && g.y > 0)
        pw += prefill_work(A, g.y, g.w, cached ? c_mode[s].y : W.segs[s].window);
    }
    const bool big = block_sum(pw, s_fsum) >= kPrefillMinWork;
    int64_t n1 = 0, n2 = 0, nrows = 0;  // units on routes 1 and 2, packed rows of live segments
    for (int64_t s = sa; s < sb; ++s) {
      const int32_t bits = bits_of((int)s);
      const int fl = flag[s];
      if (bits == 0 && fl) atomicOr(&s_status, SDPA_SEG_OVERLAP);
      const int4 g = seg_of((int)s);
      int route = kRouteNone, nrb = 0;
      if (bits == 0 && !fl && g.y > 0) {
        const int64_t R = (int64_t)g.y * A.group;
        route = route_of(A, g.y, big);
        const int rpu = rows_per_unit(A, route);
        nrb = (int)udiv(R + rpu - 1, rpu);
        if (route == kRouteSplitk) n1 += (int64_t)A.Hkv * nrb; else n2 += (int64_t)A.Hkv * nrb;
        nrows += g.y;
      }
      if (cached) {
        c_rn[s] = make_int2(route, nrb);
      } else {
        W.segs[s].route = route;
        W.segs[s].nrb = nrb;
      }
    }
    {
      int64_t cnt[3] = {n1, n2, nrows}, tot[3];
      block_scan<3>(cnt, tot, sh);
      n1 = cnt[0];
      n2 = cnt[1];
      // Live segments cover disjoint rows, so tot <= unit_cap; units past the cap (none)
      // would simply not be generated.
      if (threadIdx.x == 0) {
        s_U[1] = min(tot[0], W.unit_cap[1]);
        s_U[2] = min(tot[1], W.unit_cap[2]);
        if (tot[2] < T) s_work = 1;  // rows no live segment covers: the combine pass zeroes them
      }
    }
    for (int64_t s = sa; s < sb; ++s) {
      int2 rn;
      if (cached) {
        c_ub[s] = make_int2((int32_t)n1, (int32_t)n2);
        rn = c_rn[s];
      } else {
        W.segs[s].ubase[1] = (int32_t)n1;
        W.segs[s].ubase[2] = (int32_t)n2;
        rn = make_int2(W.segs[s].route, W.segs[s].nrb);
      }
      if (rn.x == kRouteSplitk) n1 += (int64_t)A.Hkv * rn.y;
      else if (rn.x == kRoutePrefill) n2 += (int64_t)A.Hkv * rn.y;
    }
    __syncthreads();
  }

  // 4-6. the units of both routes in one index space, [0, U1) on route 1 and [U1, U1 + U2) on
  // route 2: records, key tiles and re-read bytes, then each unit's place on its route's tile
  // line, its phase and its stream-K split
  const int64_t U1 = s_U[1], U2 = s_U[2], U = U1 + U2;
  // phases each route may use: every phase adds at most G - 1 (unit, CTA) pairs to the one
  // pair per unit, and the partial slots hold units + kPartPhases * G pairs
  constexpr int64_t kPhases = kPartPhases < kMaxPhases ? kPartPhases : kMaxPhases;
  // owning segment of unit uq of route q: the last one whose route-q unit base is <= uq
  auto owner = [&](int q, int64_t uq) -> int {
    int lo = 0, hi = S - 1, s = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int32_t ubm = cached ? (q == 1 ? c_ub[mid].x : c_ub[mid].y) : W.segs[mid].ubase[q];
      if (ubm <= uq) { s = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    return s;
  };
  auto view_of = [&](int s, int q) -> SegView {
    SegView g;
    if (cached) {
      const int4 c = c_seg[s];
      g.q_start = c.x; g.q_len = c.y; g.col = c.z; g.kv_end = c.w;
      g.nrb = c_rn[s].y;
      g.ubase = q == 1 ? c_ub[s].x : c_ub[s].y;
      g.causal = c_mode[s].x;
      g.window = c_mode[s].y;
    } else {
      const SegRec& r = W.segs[s];
      g.q_start = r.q_start; g.q_len = r.q_len; g.col = r.col; g.kv_end = r.kv_end;
      g.nrb = r.nrb;
      g.ubase = q == 1 ? r.ubase[1] : r.ubase[2];
      g.causal = r.causal;
      g.window = r.window;
    }
    return g;
  };
  const bool units_cached = U <= kUnitCache;
  {
    UnitRec* ubuf1 = units_cached ? c_unit : W.units[1];
    UnitRec* ubuf2 = units_cached ? c_unit + U1 : W.units[2];
    auto unit_at = [&](int64_t u) -> UnitRec& { return u < U1 ? ubuf1[u] : ubuf2[u - U1]; };
    int64_t ua, ub;
    my_range(U, &ua, &ub);
    // 4. records; the span and the re-read bytes wait in tile_base and slot_base
    int64_t t1 = 0, t2 = 0, b1 = 0, b2 = 0;  // key-line tiles and re-read bytes on routes 1, 2
    for (int64_t u = ua; u < ub; ++u) {
      const int q = u < U1 ? 1 : 2;
      const int64_t uq = q == 1 ? u : u - U1;
      const int s = owner(q, uq);
      int64_t span, reuse;
      UnitRec ur = make_unit(A, s, view_of(s, q), q, uq, &span, &reuse);
      if (ur.ntiles == 0) s_work = 1;  // rows of a unit with no keys: zeroed by the combine pass
      if (q == kRouteSplitk) W.unit_done[uq] = 0;
      ur.tile_base = span;
      ur.slot_base = reuse;
      unit_at(u) = ur;
      if (q == 1) {
        t1 += span;
        b1 += reuse;
      } else {
        t2 += span;
        b2 += reuse;
      }
    }
    int64_t tot4[4];
    {
      int64_t v[4] = {t1, t2, b1, b2};
      block_scan<4>(v, tot4, sh);
      t1 = v[0]; t2 = v[1]; b1 = v[2]; b2 = v[3];
    }
    for (int64_t u = ua; u < ub; ++u) {
      const bool r1 = u < U1;
      UnitRec& ur = unit_at(u);
      const int64_t span = ur.tile_base, reuse = ur.slot_base;
      int64_t& tt = r1 ? t1 : t2;
      int64_t& bb = r1 ? b1 : b2;
      ur.tile_base = tt;
      ur.phase = phase_of(bb, (int)kPhases - 1);
      tt += span;
      bb += reuse;
    }
    __syncthreads();

    // 5. phase bases: phase k of a route starts at the first unit whose phase is >= k; each
    // phase's longest unit span
    for (int64_t u = ua; u < ub; ++u) {
      const int q = u < U1 ? 1 : 2;
      const int64_t uq = q == 1 ? u : u - U1;
      const UnitRec& ur = unit_at(u);
      const int cp = ur.phase, pp = uq > 0 ? unit_at(u - 1).phase : -1;
      for (int k = pp + 1; k <= cp; ++k) {
        s_pb[q][k] = ur.tile_base;
        s_pu0[q][k] = uq;
      }
      if (ur.ntiles > 0)
        atomicMax(&s_pmax[q][cp], (int32_t)(ur.ntiles * tile_cost(q, ur.rows) + lead_cost(q)));
    }
    if (threadIdx.x < 2) {
      const int q = 1 + threadIdx.x;
      const int64_t Uq = s_U[q];
      const int64_t np = Uq > 0 ? unit_at(q == 1 ? Uq - 1 : U1 + Uq - 1).phase + 1 : 0;
      s_np[q] = np;
      s_pb[q][0] = 0;
      s_pu0[q][0] = 0;
      s_pb[q][np] = q == 1 ? tot4[0] : tot4[1];
      s_pu0[q][np] = Uq;
    }
    __syncthreads();

    // 6. stream-K within each phase, then each split unit's first partial row
    int64_t p1 = 0, p2 = 0;  // partial rows on routes 1, 2
    for (int64_t u = ua; u < ub; ++u) {
      const int q = u < U1 ? 1 : 2;
      const int64_t uq = q == 1 ? u : u - U1;
      UnitRec& ur = unit_at(u);
      const int64_t pr = place_unit(A, ur, q, uq, s_pb[q], s_pu0[q],
                                    phase_is_aligned(s_pb[q], s_pu0[q], s_pmax[q], ur.phase, A.grid[q], q));
      if (ur.nslots > 1) s_work = 1;  // split units the combine pass merges
      (q == 1 ? p1 : p2) += pr;
    }
    {
      int64_t v[2] = {p1, p2}, tot[2];
      block_scan<2>(v, tot, sh);
      p1 = v[0];
      p2 = v[1];
    }
    for (int64_t u = ua; u < ub; ++u) {
      const int q = u < U1 ? 1 : 2;
      UnitRec& ur = unit_at(u);
      int64_t& pp = q == 1 ? p1 : p2;
      ur.slot_base = pp;
      if (ur.nslots > 1) pp += (int64_t)ur.nslots * ur.rows;
    }
  }
  __syncthreads();

  // 7. write the shared-memory records out, then the header
  if (units_cached) {
    const int4* src = reinterpret_cast<const int4*>(c_unit);
    constexpr int kWords = (int)(sizeof(UnitRec) / 16);
    for (int64_t i = threadIdx.x; i < U * kWords; i += blockDim.x) {
      int4* dst = i < U1 * kWords ? reinterpret_cast<int4*>(W.units[1]) + i
                                  : reinterpret_cast<int4*>(W.units[2]) + (i - U1 * kWords);
      *dst = src[i];
    }
  }
  if (cached) {
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
      const int4 c = c_seg[s];
      SegRec r;
      r.q_start = c.x; r.q_len = c.y; r.col = c.z; r.kv_end = c.w;
      r.route = c_rn[s].x; r.nrb = c_rn[s].y; r.bits = c_bits[s]; r.pad = 0;
      r.ubase[0] = 0; r.ubase[1] = c_ub[s].x; r.ubase[2] = c_ub[s].y; r.ubase[3] = 0;
      r.causal = c_mode[s].x; r.window = c_mode[s].y;
      r.pad2[0] = r.pad2[1] = 0;
      W.segs[s] = r;
    }
  }
  // each packed row's owner as the combine pass needs it, so that it reaches the row's unit
  // in one load
  for (int64_t t = threadIdx.x; t < T; t += blockDim.x) {
    const int s = row_map[t];
    int4 ri = make_int4(kRouteNone, 0, 0, 0);
    if (s >= 0) {
      int route, nrb, ub, qs;
      if (cached) {
        route = c_rn[s].x;
        nrb = c_rn[s].y;
        ub = route == kRouteSplitk ? c_ub[s].x : c_ub[s].y;
        qs = c_seg[s].x;
      } else {
        const SegRec& r = W.segs[s];
        route = r.route;
        nrb = r.nrb;
        ub = route == kRouteSplitk ? r.ubase[kRouteSplitk] : r.ubase[kRoutePrefill];
        qs = r.q_start;
      }
      if (route != kRouteNone) ri = make_int4(route, ub, nrb, (int)(t - qs));
    }
    W.row_info[t] = ri;
  }
  for (int i = threadIdx.x; i < 2 * (kMaxPhases + 1); i += blockDim.x) {
    const int q = 1 + i / (kMaxPhases + 1), k = i % (kMaxPhases + 1);
    if (k <= s_np[q]) {
      W.hdr->phase_base[q][k] = s_pb[q][k];
      W.hdr->phase_unit0[q][k] = s_pu0[q][k];
    }
  }
  if (threadIdx.x < 2) {
    const int q = 1 + threadIdx.x;
    int64_t am = 0;
    for (int k = 0; k < s_np[q]; ++k)
      if (phase_is_aligned(s_pb[q], s_pu0[q], s_pmax[q], k, A.grid[q], q)) am |= (int64_t)1 << k;
    W.hdr->aligned[q] = am;
    W.hdr->tiles[q] = s_pb[q][s_np[q]];
    W.hdr->units[q] = s_U[q];
    W.hdr->grid[q] = A.grid[q];
    W.hdr->nphase[q] = s_np[q];
  }
  if (threadIdx.x == 0) {
    W.hdr->combine_work = s_work;
    W.hdr->status = s_status;
    if (A.status_dev && s_status) atomicOr(A.status_dev, s_status);
  }
}


// Scheduler for small calls (sched_small_ok: at most 32 segments, units one per thread): the
// records of the kernel above, from a short chain in compact code.  The scheduler runs once
// per call, from a cold instruction cache (the attention kernels ran in between), so its
// time is mostly the instruction fetch along the path it takes and the dependent steps on
// that path:
//   - warp 0 validates the segments (one per lane), tests them for shared rows with
//     shuffles (one test when the live segments are in row order, else every pair), routes
//     them and scans the unit bases, while the other warps clear the row records;
//   - after one barrier, warps take the live segments' row records and every thread one
//     unit: its record, then two scans over the warps of its route (route 2's units start
//     at a warp boundary, so a warp holds one route) with one barrier each, and one barrier
//     for the phase bases, which each thread writes for the next unit of its route from its
//     own prefix and span.
__global__ void __launch_bounds__(kSchedThreads) sdpa_sched_small_kernel(SchedArgs A) {
  __shared__ int4 c_seg[kSmallSegs];   // (q_start, q_len, col, kv_end)
  __shared__ int2 c_mode[kSmallSegs];  // (causal, window)
  __shared__ int2 c_rn[kSmallSegs];    // (route, nrb)
  __shared__ int2 c_ub[kSmallSegs];    // unit bases on routes 1 and 2
  __shared__ int64_t sh[3 * 32];
  __shared__ int64_t s_pb[3][kMaxPhases + 1];
  __shared__ int64_t s_pu0[3][kMaxPhases + 1];  // first unit of each phase; [np] = units
  __shared__ int32_t s_pmax[3][kMaxPhases];      // longest unit span of each phase
  __shared__ int32_t s_U[3], s_np[3], s_status, s_work;
  const Workspace& W = A.ws;
  const int S = A.S;
  const int T = (int)A.T;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  constexpr uint32_t kAll = 0xffffffffu;

  if (warp == 0) {
    const bool have = lane < S;
    int32_t g[4] = {0, 0, 0, 0};
    int2 md = make_int2(A.causal, A.window);
    if (have) {
      load_seg(A, lane, g);
      if (A.seg_mode) md = reinterpret_cast<const int2*>(A.seg_mode)[lane];
    }
    // the attention kernels may start launching (they wait for this grid); the trigger takes
    // a while, and the loads above are in flight meanwhile
    griddep_launch();
    md.x = md.x != 0;
    const int32_t bits = have ? segment_bits(g[0], g[1], g[2], g[3], T, A.rows, A.cols, md.y) : 0;
    const bool ok = have && bits == 0 && g[1] > 0;
    const uint32_t okm = __ballot_sync(kAll, ok);
    // a valid segment that shares a packed row with another valid one: both are dropped
    const int32_t a0 = ok ? g[0] : 0, a1 = ok ? g[0] + g[1] : 0;  // in [0, T] when ok
    const int nxt = __ffs(okm & ~((2u << lane) - 1u)) - 1;       // next valid lane, or -1
    const int32_t n0 = __shfl_sync(kAll, a0, nxt < 0 ? lane : nxt);
    bool ov = false;
    if (!__all_sync(kAll, !ok || nxt < 0 || a1 <= n0)) {
#pragma unroll 1
      for (int o = 0; o < kSmallSegs; ++o) {
        const int32_t b0 = __shfl_sync(kAll, a0, o), b1 = __shfl_sync(kAll, a1, o);
        ov |= o != lane && ((okm >> o) & 1u) && max(a0, b0) < min(a1, b1);
      }
      ov = ov && ok;
    }
    const bool live = ok && !ov;
    float pw = live ? prefill_work(A, g[1], g[3], md.y) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pw += __shfl_xor_sync(kAll, pw, o);
    int route = kRouteNone, nrb = 0;
    if (live) {
      route = route_of(A, g[1], pw >= kPrefillMinWork);
      const int rpu = rows_per_unit(A, route);
      nrb = (int)(((uint32_t)g[1] * (uint32_t)A.group + rpu - 1) / (uint32_t)rpu);
    }
    const int32_t n1 = route == kRouteSplitk ? A.Hkv * nrb : 0, n2 = route == kRoutePrefill ? A.Hkv * nrb : 0;
    int32_t x1 = n1, x2 = n2;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y1 = __shfl_up_sync(kAll, x1, o), y2 = __shfl_up_sync(kAll, x2, o);
      if (lane >= o) {
        x1 += y1;
        x2 += y2;
      }
    }
    const int32_t covered = (int32_t)__reduce_add_sync(kAll, live ? (uint32_t)g[1] : 0u);
    const int32_t st = (int32_t)__reduce_or_sync(kAll, (uint32_t)(bits | (ov ? SDPA_SEG_OVERLAP : 0)));
    if (have) {
      c_seg[lane] = make_int4(g[0], g[1], g[2], g[3]);
      c_mode[lane] = md;
      c_rn[lane] = make_int2(route, nrb);
      c_ub[lane] = make_int2(x1 - n1, x2 - n2);
      SegRec r;
      r.q_start = g[0]; r.q_len = g[1]; r.col = g[2]; r.kv_end = g[3];
      r.route = route; r.nrb = nrb; r.bits = bits; r.pad = 0;
      r.ubase[0] = 0; r.ubase[1] = x1 - n1; r.ubase[2] = x2 - n2; r.ubase[3] = 0;
      r.causal = md.x; r.window = md.y;
      r.pad2[0] = r.pad2[1] = 0;
      W.segs[lane] = r;
    }
    if (lane == 31) {
      s_status = st;
      s_work = covered < T;  // rows no live segment covers: the combine pass zeroes them
      s_U[1] = (int32_t)min((int64_t)x1, W.unit_cap[1]);
      s_U[2] = (int32_t)min((int64_t)x2, W.unit_cap[2]);
    }
  } else {
    griddep_launch();
    if (threadIdx.x - 32 < 3 * kMaxPhases) (&s_pmax[0][0])[threadIdx.x - 32] = 0;
    for (int t = threadIdx.x - 32; t < T; t += blockDim.x - 32) W.row_info[t] = make_int4(kRouteNone, 0, 0, 0);
  }
  __syncthreads();  // (also orders the row records above before the ones below)

  // each live segment's row records
  for (int s = warp; s < S; s += nw) {
    const int2 rn = c_rn[s];
    if (rn.x == kRouteNone) continue;
    const int4 g = c_seg[s];
    const int ub = rn.x == kRouteSplitk ? c_ub[s].x : c_ub[s].y;
    for (int i = lane; i < g.y; i += 32) W.row_info[g.x + i] = make_int4(rn.x, ub, rn.y, i);
  }

  // one unit per thread
  const int U1 = s_U[1], U2 = s_U[2], U1w = (U1 + 31) & ~31;
  constexpr int kPhases = kPartPhases < kMaxPhases ? kPartPhases : kMaxPhases;
  const int i = threadIdx.x;
  const int q = i < U1 ? 1 : (i >= U1w && i < U1w + U2 ? 2 : 0);
  const int uq = q == 1 ? i : i - U1w;
  auto wroute = [&](int w) -> int {
    const int w0 = w * 32;
    return w0 < U1 ? 1 : (w0 >= U1w && w0 < U1w + U2 ? 2 : 0);
  };
  UnitRec ur;
  int64_t span = 0, reuse = 0;
  if (q != 0) {
    // owning segment: the last one whose route-q unit base is <= uq
    int lo = 0, hi = S - 1, s = 0;
#pragma unroll 1
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if ((q == 1 ? c_ub[mid].x : c_ub[mid].y) <= uq) { s = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    const int4 c = c_seg[s];
    SegView gv;
    gv.q_start = c.x; gv.q_len = c.y; gv.col = c.z; gv.kv_end = c.w;
    gv.nrb = c_rn[s].y;
    gv.ubase = q == 1 ? c_ub[s].x : c_ub[s].y;
    gv.causal = c_mode[s].x;
    gv.window = c_mode[s].y;
    ur = make_unit(A, s, gv, q, uq, &span, &reuse);
    if (ur.ntiles == 0) s_work = 1;  // rows of a unit with no keys: zeroed by the combine pass
    if (q == kRouteSplitk) W.unit_done[uq] = 0;
  }
  int64_t v[2] = {span, reuse}, tot[2];
  route_scan<2>(v, tot, sh, wroute);
  if (q != 0) {
    const int64_t tb = v[0], bb = v[1];
    ur.tile_base = tb;
    ur.phase = phase_of(bb, kPhases - 1);
    atomicMax(&s_pmax[q][ur.phase], (int32_t)span);
    if (uq == 0) {
      s_pb[q][0] = 0;
      s_pu0[q][0] = 0;
    }
    if (uq + 1 < (q == 1 ? U1 : U2)) {
      const int pn = phase_of(bb + reuse, kPhases - 1);
      for (int k = ur.phase + 1; k <= pn; ++k) {
        s_pb[q][k] = tb + span;
        s_pu0[q][k] = uq + 1;
      }
    } else {
      s_np[q] = ur.phase + 1;
      s_pb[q][ur.phase + 1] = tot[0];
      s_pu0[q][ur.phase + 1] = uq + 1;
    }
  }
  if (i < 2 && s_U[1 + i] == 0) {
    s_np[1 + i] = 0;
    s_pb[1 + i][0] = 0;
    s_pu0[1 + i][0] = 0;
  }
  __syncthreads();
  int64_t pv[1] = {0}, ptot[1];
  if (q != 0) {
    pv[0] = place_unit(A, ur, q, uq, s_pb[q], s_pu0[q],
                       phase_is_aligned(s_pb[q], s_pu0[q], s_pmax[q], ur.phase, A.grid[q], q));
    if (ur.nslots > 1) s_work = 1;  // split units the combine pass merges
  }
  route_scan<1>(pv, ptot, sh + 2 * 32, wroute);  // (its barrier also publishes s_work)
  if (q != 0) {
    ur.slot_base = pv[0];
    W.units[q][uq] = ur;
  }

  // the header
  if (i < 2 * (kMaxPhases + 1)) {
    const int hq = 1 + i / (kMaxPhases + 1), k = i % (kMaxPhases + 1);
    if (k <= s_np[hq]) {
      W.hdr->phase_base[hq][k] = s_pb[hq][k];
      W.hdr->phase_unit0[hq][k] = s_pu0[hq][k];
    }
  }
  if (i < 2) {
    const int hq = 1 + i;
    int64_t am = 0;
    for (int k = 0; k < s_np[hq]; ++k)
      if (phase_is_aligned(s_pb[hq], s_pu0[hq], s_pmax[hq], k, A.grid[hq], hq)) am |= (int64_t)1 << k;
    W.hdr->aligned[hq] = am;
    W.hdr->tiles[hq] = s_pb[hq][s_np[hq]];
    W.hdr->units[hq] = s_U[hq];
    W.hdr->grid[hq] = A.grid[hq];
    W.hdr->nphase[hq] = s_np[hq];
  }
  if (i == 0) {
    W.hdr->combine_work = s_work;
    W.hdr->status = s_status;
    if (A.status_dev && s_status) atomicOr(A.status_dev, s_status);
  }
}

const void* sched_kernel_ptr() { return (const void*)sdpa_sched_kernel; }
const void* sched_small_kernel_ptr() { return (const void*)sdpa_sched_small_kernel; }

cudaError_t launch_sched(const SchedArgs& sa, cudaStream_t st) {
  void* args[] = {(void*)&sa};
  if (sched_small_ok(sa.T, sa.group * sa.Hkv, sa.Hkv, sa.S))
    return cudaLaunchKernel(sched_small_kernel_ptr(), dim3(1), dim3(kSchedThreads), args, 0, st);
  return cudaLaunchKernel(sched_kernel_ptr(), dim3(1), dim3(kSchedThreads), args, sched_smem_bytes(), st);
}
size_t sched_smem_bytes() { return kSchedSmem; }

}  // namespace sdpa
