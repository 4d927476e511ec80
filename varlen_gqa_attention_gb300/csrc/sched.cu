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
//      all units' tiles end to end, each unit's behind a few placeholder tiles for the cost
//      of starting a piece; the line is cut into at most four phases whose re-read K/V fits
//      the L2 budget; within a phase CTA g of G owns tiles [g*W/G, (g+1)*W/G) (a stream-K
//      split, so every CTA gets the same amount of key tiles whatever the length mix; G is
//      capped at W so that no CTA is idle inside a unit's range), the CTAs whose share
//      starts in a unit are recorded against it, and each (unit, CTA) pair gets a slot of
//      partial results unless the unit has a single CTA, which then writes `out` itself;
//   5. publishes the records, a per-row record for the combine pass, the arrival counters
//      of the split units (zeroed) and a flag that tells the combine pass whether it has
//      any work.
// One CTA of 512 threads does all of it; block-wide scans give the prefix sums.  Segment
// tables of up to 1024 segments, up to 8192 packed rows and up to 1024 units are built in
// shared memory; larger calls run the same steps on the workspace copies.
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
// Start-up cost of a piece in key tiles of its route (operand loads, pipeline fill, the
// epilogue): about 4 us per prefill piece of 128-key tiles that take about 0.7 us, about
// 4 us per split-K piece of 64-key tiles that stream at about 1.6 us.
__device__ __forceinline__ int64_t lead_tiles(int route) { return route == kRoutePrefill ? 6 : 3; }

// Route of a live segment.  The prefill kernel takes segments that fill at least one
// 128-row tile (on a ring store too: its key tiles stop at the wrap, so a TMA box never
// wraps); everything else, and everything when the prefill kernel is unusable, goes to the
// split-K kernel.
__device__ __forceinline__ int route_of(const SchedArgs& A, const SegRec& r) {
  const int64_t R = (int64_t)r.q_len * A.group;
  if (A.policy == SDPA_ROUTE_SPLITK || !A.prefill_ok) return kRouteSplitk;
  if (A.policy == SDPA_ROUTE_PREFILL) return kRoutePrefill;
  return R >= kPrefillRows ? kRoutePrefill : kRouteSplitk;
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
  __shared__ int64_t s_pb[3][kMaxPhases + 1];
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
  griddep_launch();  // the attention kernels may start launching; they wait for this grid
  if (threadIdx.x == 0) {
    s_status = 0;
    s_work = 0;
  }
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
  auto seg_of = [&](int s) -> int4 {
    if (cached) return c_seg[s];
    const SegRec r = W.segs[s];
    return make_int4(r.q_start, r.q_len, r.col, r.kv_end);
  };
  auto bits_of = [&](int s) -> int32_t { return cached ? c_bits[s] : W.segs[s].bits; };

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
  // the finished owner map goes out for the combine pass
  int64_t sa, sb;
  my_range(S, &sa, &sb);
  int64_t n1 = 0, n2 = 0, nrows = 0;  // units on routes 1 and 2, packed rows of live segments
  for (int64_t s = sa; s < sb; ++s) {
    const int32_t bits = bits_of((int)s);
    const int fl = flag[s];
    if (bits == 0 && fl) atomicOr(&s_status, SDPA_SEG_OVERLAP);
    const int4 g = seg_of((int)s);
    int route = kRouteNone, nrb = 0;
    if (bits == 0 && !fl && g.y > 0) {
      SegRec r;
      r.q_start = g.x; r.q_len = g.y; r.col = g.z; r.kv_end = g.w;
      r.window = cached ? c_mode[s].y : W.segs[s].window;
      const int64_t R = (int64_t)g.y * A.group;
      route = route_of(A, r);
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

  // 4. the units of both routes in one index space, [0, U1) on route 1 and [U1, U1 + U2) on
  // route 2, each thread a contiguous range: records, key tiles and re-read bytes, then
  // each unit's place on its route's tile line and its phase
  const int64_t U1 = s_U[1], U2 = s_U[2], U = U1 + U2;
  const bool units_cached = U <= kUnitCache;
  UnitRec* ubuf1 = units_cached ? c_unit : W.units[1];
  UnitRec* ubuf2 = units_cached ? c_unit + U1 : W.units[2];
  auto unit_at = [&](int64_t u) -> UnitRec& { return u < U1 ? ubuf1[u] : ubuf2[u - U1]; };
  // phases each route may use: every phase adds at most G - 1 (unit, CTA) pairs to the one
  // pair per unit, and the partial slots hold units + kPartPhases * G pairs
  constexpr int64_t kPhases = kPartPhases < kMaxPhases ? kPartPhases : kMaxPhases;
  int64_t ua, ub;
  my_range(U, &ua, &ub);
  int64_t t1 = 0, t2 = 0, b1 = 0, b2 = 0;  // key-line tiles and re-read bytes on routes 1, 2
  for (int64_t u = ua; u < ub; ++u) {
    const int q = u < U1 ? 1 : 2;
    const int64_t uq = q == 1 ? u : u - U1;
    const int rpu = rows_per_unit(A, q), tl = tile_len(A, q);
    // owning segment: the last one whose route-q unit base is <= uq
    int lo = 0, hi = S - 1, s = 0;
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      const int32_t ubm = cached ? (q == 1 ? c_ub[mid].x : c_ub[mid].y) : W.segs[mid].ubase[q];
      if (ubm <= uq) { s = mid; lo = mid + 1; } else { hi = mid - 1; }
    }
    struct {
      int32_t q_start, q_len, col, kv_end, nrb, ubase, causal, window;
    } g;
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
    if (nt == 0) s_work = 1;  // rows of a unit with no keys: zeroed by the combine pass
    ur.nslots = 0;
    ur.g_first = 0;
    ur.ntiles = (int32_t)nt;
    ur.phase = 0;
    const int64_t span_tiles = nt > 0 ? nt + lead_tiles(q) : 0;
    ur.tile_base = span_tiles;  // the span, until the scan below
    // K/V bytes the group's units read again (counted once, on the group's last unit;
    // only groups of several units re-read them): phases are cut on these
    int64_t reuse = 0;
    if (g.nrb >= 2 && ur.rb == g.nrb - 1) {
      int64_t span = g.kv_end;
      if (g.window > 0) span = min(span, (int64_t)g.q_len + g.window - 1);
      reuse = span * (int64_t)A.D * 4;
    }
    ur.slot_base = reuse;  // kept here until the phase pass below
    unit_at(u) = ur;
    if (q == 1) {
      t1 += span_tiles;
      b1 += reuse;
    } else {
      t2 += span_tiles;
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
    ur.phase = (int32_t)min(bb / kPhaseBytes, kPhases - 1);
    tt += span;
    bb += reuse;
  }
  __syncthreads();

  // 5. phase bases: phase k of a route starts at the first unit whose phase is >= k
  for (int64_t u = ua; u < ub; ++u) {
    const int q = u < U1 ? 1 : 2;
    const int64_t uq = q == 1 ? u : u - U1;
    const int cp = unit_at(u).phase, pp = uq > 0 ? unit_at(u - 1).phase : -1;
    for (int k = pp + 1; k <= cp; ++k) s_pb[q][k] = unit_at(u).tile_base;
  }
  if (threadIdx.x < 2) {
    const int q = 1 + threadIdx.x;
    const int64_t Uq = s_U[q];
    const int64_t np = Uq > 0 ? unit_at(q == 1 ? Uq - 1 : U1 + Uq - 1).phase + 1 : 0;
    s_np[q] = np;
    s_pb[q][0] = 0;
    s_pb[q][np] = q == 1 ? tot4[0] : tot4[1];
  }
  __syncthreads();

  // 6. stream-K within each phase: CTA g of G_p = min(G, W_p) owns [g W_p / G_p, (g+1) W_p / G_p);
  // G_p <= W_p makes every working CTA own a tile, so the owners of a unit's tiles are
  // consecutive CTAs that all work on it (nslots is exact)
  int64_t p1 = 0, p2 = 0;  // partial rows on routes 1, 2
  for (int64_t u = ua; u < ub; ++u) {
    const int q = u < U1 ? 1 : 2;
    const int64_t uq = q == 1 ? u : u - U1;
    UnitRec& ur = unit_at(u);
    const int64_t nt = ur.ntiles;
    if (nt > 0) {
      const int64_t G = A.grid[q];
      const int64_t lead = lead_tiles(q);
      const int64_t b0 = s_pb[q][ur.phase];
      const int64_t Wp = s_pb[q][ur.phase + 1] - b0;
      const int64_t Gp = min(G, Wp);
      const int64_t k0 = ur.tile_base + lead - b0;  // the key tiles, phase-relative
      const int64_t g0 = sk_owner(k0, Wp, Gp);
      const int64_t g1 = sk_owner(k0 + nt - 1, Wp, Gp);
      ur.g_first = (int32_t)g0;
      ur.nslots = (int32_t)(g1 - g0 + 1);
      if (ur.nslots > 1) (q == 1 ? p1 : p2) += (int64_t)ur.nslots * ur.rows;
      // split units the combine pass merges
      if (ur.nslots > 1) s_work = 1;
      // CTAs whose share starts inside this unit's span begin their walk here: the ones
      // after the owner of the tile before the span, up to the owner of its last tile
      const int64_t s0 = ur.tile_base - b0, s1 = k0 + nt;
      const int64_t c0 = s0 > 0 ? sk_owner(s0 - 1, Wp, Gp) + 1 : 0;
      for (int64_t c = c0; c <= sk_owner(s1 - 1, Wp, Gp); ++c) W.first_unit[q][ur.phase * G + c] = (int32_t)uq;
    }
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
    if (k <= s_np[q]) W.hdr->phase_base[q][k] = s_pb[q][k];
  }
  if (threadIdx.x < 2) {
    const int q = 1 + threadIdx.x;
    W.hdr->tiles[q] = s_pb[q][s_np[q]];
    W.hdr->units[q] = s_U[q];
    W.hdr->grid[q] = A.grid[q];
    W.hdr->lead[q] = lead_tiles(q);
    W.hdr->nphase[q] = s_np[q];
  }
  if (threadIdx.x == 0) {
    W.hdr->combine_work = s_work;
    W.hdr->status = s_status;
    if (A.status_dev && s_status) atomicOr(A.status_dev, s_status);
  }
}

const void* sched_kernel_ptr() { return (const void*)sdpa_sched_kernel; }
size_t sched_smem_bytes() { return kSchedSmem; }

}  // namespace sdpa
