// common.cuh - shared definitions of the sm_103a attention kernels: workspace layout,
// segment/unit records written by the device scheduler, and small inline-PTX helpers.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdpa_varlen.h"

namespace sdpa {

// Rows of one work unit: query rows (t, g) packed as r = i * group + g, so the query
// heads that share a KV head sit side by side in one tile (GQA packing).
// split-K kernel: up to two 16-row groups, the four warps splitting each key tile among
// them; more rows per unit would leave each warp a whole tile of legacy tensor-core work
constexpr int kSplitkRows = 32;
constexpr int kSplitkTile = 64;    // split-K kernel: key positions per tile
constexpr int kSplitkThreads = 128;  // split-K kernel: four warps
constexpr int kPrefillRows = 128;  // tensor-memory prefill kernel: one 128-lane accumulator
// The prefill route is taken only by a call whose segments of at least kPrefillRows packed
// rows hold this much work, measured as sum(packed rows * needed key span) * Hkv * D: below
// it the tensor-memory kernel's fixed cost (set-up, first loads, epilogue: ~15 us) is more
// than the split-K kernel's extra time (measured crossover: ~2^30 at D = 64 and D = 128,
// about 2 GFLOP of causal work).
constexpr float kPrefillMinWork = 1073741824.0f;
constexpr int kPrefillTile = 128;  // prefill kernel: key positions per tile
// Packed rows of a prefill unit: two 128-row halves that share every K/V tile (D = 64, 128),
// or one (D = 256, whose output accumulator alone fills the tensor memory).
__host__ __device__ constexpr int prefill_unit_rows(int D) { return D == 256 ? kPrefillRows : 2 * kPrefillRows; }

constexpr int kRouteNone = 0;
constexpr int kRouteSplitk = 1;
constexpr int kRoutePrefill = 2;

// Per-segment record (the scheduler's view of one seq_info row).
struct SegRec {
  int32_t q_start, q_len, col, kv_end;
  int32_t route;     // kRoute*: none for invalid, overlapping or empty segments
  int32_t nrb;       // row blocks per KV head (units per KV head)
  int32_t bits;      // SDPA_SEG_* bits of this segment
  int32_t pad;
  int32_t ubase[4];  // per route: units of all earlier segments on that route (monotone in
                     // the segment index, so a binary search maps a unit to its segment)
  int32_t causal, window;  // the segment's mask mode (the call's, or its row of seg_mode)
  int32_t pad2[2];
};

// Per-unit record: (segment, KV head, row block) and its stream-K split.
struct UnitRec {
  int32_t seg, hk, rb, rows;  // rows = query rows in this unit (<= unit size)
  int32_t lo, hi;             // key positions the unit's rows see together: [lo, hi)
  int32_t nslots;             // CTAs that work on the unit (0: no keys; 1: written directly)
  int32_t g_first;            // first such CTA
  int32_t ntiles;             // key tiles of the unit
  int32_t phase;              // scheduling phase of the unit (see SchedHdr)
  int32_t q_start, q_len, col, kv_end;  // the segment's entry and mask mode, copied so
  int32_t causal, window;               // that one record (80 bytes) describes a piece
  int64_t tile_base;          // start of the unit's span on its route's line of cost units:
                              // lead_cost placeholders, then its ntiles key tiles
  int64_t slot_base;          // first partial row of the unit's slots
};
static_assert(sizeof(UnitRec) == 80, "unit record layout");


// Phases: a route's tile line is cut at (segment, KV head) boundaries into phases whose
// re-read K/V (units sharing a group's keys) fits a budget below the L2 size; every CTA
// takes its stream-K share of phase 0, then of phase 1, ... so the K/V tiles the whole
// grid touches at one time stay cached.  The header and the per-CTA start tables have room
// for kMaxPhases; the scheduler uses at most kPartPhases (the partial slots' sizing).
constexpr int kMaxPhases = 16;
constexpr int64_t kPhaseBytes = 48ll << 20;

// Scheduler header (int64 words).
struct SchedHdr {
  int64_t tiles[3];   // length of each route's line, in cost units (index = route)
  int64_t units[3];   // units per route
  int64_t grid[3];    // CTAs per route as launched
  int64_t status;     // OR of the status bits of this call
  int64_t nphase[3];  // phases per route
  int64_t phase_base[3][kMaxPhases + 1];  // start of each phase on the line; [nphase] = tiles
  // Phases of short, even units take one whole unit per CTA ("aligned": CTA g of the phase
  // works on its unit u0 + g alone, so no unit is cut and no partial slot is written; the
  // scheduler's phase_is_aligned decides); phase_unit0[p] = the phase's first unit.
  int64_t aligned[3];  // bit p: phase p is aligned
  int64_t phase_unit0[3][kMaxPhases + 1];
  // Non-zero when the combine pass has rows to write: rows no live segment covers, units
  // with no keys, or units split over several CTAs.
  int64_t combine_work;
};

struct Workspace {
  SchedHdr* hdr;
  SegRec* segs;
  int32_t* row_seg;     // [T] owning segment or -1 (the scheduler's claims)
  int4* row_info;       // [T] for the combine pass: (route, the segment's first unit on that
                        // route, units per KV head, row within the segment); route 0: no
                        // live segment owns the row
  int32_t* seg_flag;    // [S] overlap flags
  UnitRec* units[3];    // [route][U_cap]
  int32_t* first_unit[3];  // [route][phase * grid + CTA]: unit whose span holds the CTA's first tile
  float2* part_ml[3];   // [route][P_cap] (running max in log2 units, sum)
  float* part_o[3];     // [route][P_cap * D] unnormalised output
  int64_t unit_cap[3];
  int64_t part_cap[3];
  // [U_cap of the split-K route] CTAs of each split-K unit that have written their partial
  // slot (zeroed by the scheduler, counted by the split-K kernel with release semantics, read
  // by the combine pass with acquire semantics)
  int32_t* unit_done;
};

__host__ __device__ inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Units a route can produce for T packed rows in S segments (non-overlapping after the
// scheduler drops overlapping segments): sum_s ceil(q_len_s * group / R) <= T*group/R + S.
__host__ __device__ inline int64_t unit_cap(int64_t T, int Hq, int Hkv, int S, int rows_per_unit) {
  int group = Hq / Hkv;
  return (int64_t)Hkv * ((T * group) / rows_per_unit + (int64_t)S + 1);
}

// Partial rows: each (unit, CTA) pair that is not the only CTA of its unit writes one slot
// of `unit rows` rows.  Within one phase the CTAs' shares cut the units at most grid - 1
// times, so there are at most units + phases * grid pairs; the slots are sized for
// kPartPhases phases, and the scheduler uses no more.
constexpr int kPartPhases = 4;
__host__ __device__ inline int64_t part_cap(int64_t ucap, int64_t grid, int rows_per_unit) {
  return (ucap + kPartPhases * grid + 1) * rows_per_unit;
}

// Lays the workspace out from `base` (base may be null to only measure). Returns bytes.
// Without the prefill route (`with_prefill` false: every segment takes the split-K kernel)
// that route's unit table and partial slots are empty.
__host__ inline size_t layout_workspace(char* base, int64_t T, int Hq, int Hkv, int D, int S,
                                        int64_t grid_splitk, int64_t grid_prefill,
                                        Workspace* ws, bool with_prefill = true) {
  int64_t off = 0;
  auto take = [&](int64_t bytes) {
    int64_t o = off;
    off = align_up(off + bytes, 256);
    return base ? base + o : nullptr;
  };
  Workspace w{};
  w.hdr = (SchedHdr*)take(sizeof(SchedHdr));
  w.segs = (SegRec*)take((int64_t)sizeof(SegRec) * (S > 0 ? S : 1));
  w.row_seg = (int32_t*)take(4 * (T > 0 ? T : 1));
  w.row_info = (int4*)take(16 * (T > 0 ? T : 1));
  w.seg_flag = (int32_t*)take(4 * (S > 0 ? S : 1));
  const int rpu[3] = {0, kSplitkRows, prefill_unit_rows(D)};
  const int64_t grid[3] = {0, grid_splitk, grid_prefill};
  for (int r = 1; r < 3; ++r) {
    const bool used = r == kRouteSplitk || with_prefill;
    w.unit_cap[r] = used ? unit_cap(T, Hq, Hkv, S, rpu[r]) : 0;
    w.part_cap[r] = used ? part_cap(w.unit_cap[r], grid[r], rpu[r]) : 0;
    w.units[r] = (UnitRec*)take((int64_t)sizeof(UnitRec) * w.unit_cap[r]);
    w.first_unit[r] = (int32_t*)take(4 * (int64_t)kMaxPhases * (grid[r] > 0 ? grid[r] : 1));
    w.part_ml[r] = (float2*)take(8 * w.part_cap[r]);
    w.part_o[r] = (float*)take(4 * w.part_cap[r] * D);
  }
  w.unit_done = (int32_t*)take(4 * (w.unit_cap[kRouteSplitk] > 0 ? w.unit_cap[kRouteSplitk] : 1));
  if (ws) *ws = w;
  return (size_t)off;
}

// Arguments shared by the attention kernels and the combine pass.
struct AttnArgs {
  const __nv_bfloat16* q;
  int64_t q_rs, q_hs;  // element strides of q rows and heads
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int64_t rows;        // store rows
  int cols, Hkv, Hq, group, D;
  int causal, window;
  float scale_log2;    // scale * log2(e): scores are kept in base-2 units
  __nv_bfloat16* out;
  int64_t o_rs, o_hs;
  int64_t T;
  Workspace ws;
  int32_t* status_dev;
};

// Arguments of the KV append kernel (the step's new rows into the column store).
struct AppendArgs {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t new_rs, new_hs;  // element strides of the new rows and heads
  __nv_bfloat16* k_store;
  __nv_bfloat16* v_store;
  int64_t rows;
  int cols, Hkv, D;
  const SegRec* segs;      // the scheduler's segment records (route none: not live)
};
constexpr int kAppendThreads = 128;

// Arguments of the column clone kernel: store rows [0, m) of column src_col copied to dst_col.
struct CloneArgs {
  __nv_bfloat16* k_store;
  __nv_bfloat16* v_store;
  int64_t m;
  int cols, Hkv, D, src_col, dst_col;
};
constexpr int kCloneThreads = 256;

// Arguments of the scheduler kernel.
struct SchedArgs {
  const int32_t* seq_info;
  const int32_t* seg_mode;  // NULL, or [S, 2] (causal, window) per segment
  int S;
  int use_inline;  // dense entry: one segment passed by value
  int32_t inl[4];
  int64_t T, rows;
  int cols, Hkv, group, causal, window;
  int D;           // head dim (bytes of the K/V each phase holds)
  int policy;      // SDPA_ROUTE_*
  int prefill_ok;  // prefill kernel usable for this call (group divides 128, tensor maps made)
  int tile_pf;     // keys per prefill tile
  int64_t grid[3];
  Workspace ws;
  int32_t* status_dev;
};

constexpr int kSchedThreads = 512;
// Calls the small scheduler kernel takes: at most kSmallSegs segments and at most 8192 packed
// rows, and units that fit one per thread with route 2's starting at a warp boundary.  Live
// segments cover disjoint rows and a unit holds at least 32 packed rows, so the units number
// at most Hkv * (ceil(T * group / 32) + S).
constexpr int kSmallSegs = 32;
__host__ __device__ inline bool sched_small_ok(int64_t T, int Hq, int Hkv, int S) {
  if (S > kSmallSegs || T > 8192 || Hkv <= 0) return false;
  const int64_t units = (int64_t)Hkv * ((T * (Hq / Hkv) + 31) / 32 + S);
  return units + 31 <= kSchedThreads;
}

// Kernel entry points (defined in their own translation units).
const void* sched_kernel_ptr();
const void* sched_small_kernel_ptr();  // calls with sched_small_ok
// Launches the scheduler kernel that suits the call (one CTA of kSchedThreads threads).
cudaError_t launch_sched(const SchedArgs& sa, cudaStream_t st);
size_t sched_smem_bytes();  // dynamic shared memory of the scheduler kernel
const void* append_kernel_ptr();
const void* clone_kernel_ptr();
const void* splitk_kernel_ptr(int D);
int splitk_smem_bytes(int D);
const void* combine_kernel_ptr(int D);
const void* prefill_kernel_ptr(int D);
const void* prefill_pair_kernel_ptr(int D);  // D = 64, 128
int prefill_pair_smem_bytes(int D);
int prefill_pair_block_threads(int D);
int prefill_smem_bytes(int D);
int prefill_tile_keys(int D);
int prefill_block_threads(int D);
// Sets the message sdpa_last_error() returns on this thread.
void set_last_error(const char* msg);
// Argument checks shared by the attention entry points (api.cu); each sets the message of
// sdpa_last_error() and returns its code, SDPA_OK when the arguments pass.
sdpa_status check_common(int64_t T, int Hq, int Hkv, int D, int S, int64_t rows, int cols, int window,
                         float scale);
sdpa_status check_tensors(const void* q, const void* k, const void* v, void* out, const int32_t* seq_info,
                          int S, int64_t q_rs, int64_t q_hs, int64_t o_rs, int64_t o_hs);

// Segment validity (SDPA_SEG_* bits), same rule on host and device.
__host__ __device__ inline int32_t segment_bits(int64_t q_start, int64_t q_len, int64_t col,
                                                int64_t kv_end, int64_t T, int64_t rows,
                                                int64_t cols, int window) {
  int32_t bits = 0;
  if (q_len < 0 || q_start < 0 || q_start + q_len > T) bits |= SDPA_SEG_BAD_QRANGE;
  if (col < 0 || col >= cols) bits |= SDPA_SEG_BAD_COL;
  if (kv_end < 0) bits |= SDPA_SEG_BAD_KV;
  if (bits == 0 && q_len > 0 && kv_end > 0) {
    int64_t span = kv_end;
    if (window > 0) span = kv_end < q_len + window - 1 ? kv_end : q_len + window - 1;
    if (span > rows) bits |= SDPA_SEG_SPAN;
  }
  return bits;
}

// Visible key positions of query row i: [lo, hi) (hi <= lo: none).
struct RowWin {
  int32_t lo, hi;
};
__device__ __forceinline__ RowWin row_window(int i, int q_len, int kv_end, int causal, int window) {
  int p = kv_end - q_len + i;
  RowWin w;
  w.hi = causal ? min(p + 1, kv_end) : kv_end;
  w.lo = window > 0 ? max(0, p - window + 1) : 0;
  return w;
}

// Work of one CTA on one route: for each phase, its stream-K share of the phase's tiles,
// cut into pieces (one unit's consecutive tiles each).  All roles of a CTA walk the same
// sequence.
struct PieceWalk {
  const Workspace* W;
  int route;
  int64_t G;        // launched grid
  int64_t nphase;
  int64_t p;        // current phase
  int64_t t0, t1;   // remaining share of this CTA in phase p (line cost units)
  int64_t u;        // next unit to look at
  int64_t U;        // units of the route
  int64_t pb0, pb1; // phase 0's tile range, and this CTA's first unit in it (loaded early)
  int32_t fu0;
  int64_t amask;    // the route's aligned phases (bit p)
};

// a / b for a >= 0, b > 0: one 32-bit division when both fit in 32 bits (the usual case).
// On the device the 64-bit division, a long instruction sequence, is a call: kept out of
// line, it does not spread the code that runs over more instruction-cache lines.
#ifdef __CUDA_ARCH__
static __device__ __noinline__ int64_t udiv64(int64_t a, int64_t b) { return a / b; }
#endif
__host__ __device__ __forceinline__ int64_t udiv(int64_t a, int64_t b) {
  if ((((uint64_t)a | (uint64_t)b) >> 32) == 0) return (int64_t)((uint32_t)a / (uint32_t)b);
#ifdef __CUDA_ARCH__
  return udiv64(a, b);
#else
  return a / b;
#endif
}

// Key tiles of a prefill unit.  The unit's keys [lo, hi) span at most `rows` store rows, so on
// a ring store they cross a multiple of `rows` (where the store row wraps to 0) at most once;
// such a range is tiled in two parts, [lo, wrap) and [wrap, hi), so that the store rows of
// every tile are consecutive (one TMA box).  The tile that ends at the wrap may be short.
struct KeyTiles {
  int64_t lo, wrap, hi;  // wrap = hi when the range does not wrap
  int64_t na, n;         // tiles of [lo, wrap), and of the whole range
};
__host__ __device__ inline KeyTiles key_tiles(int64_t lo, int64_t hi, int64_t rows, int bn) {
  KeyTiles k;
  k.lo = lo;
  k.hi = hi;
  if (hi <= lo) {
    k.wrap = hi;
    k.na = k.n = 0;
    return k;
  }
  const int64_t w = (udiv(lo, rows) + 1) * rows;  // first position after lo in store row 0
  k.wrap = w < hi ? w : hi;
  k.na = udiv(k.wrap - lo + bn - 1, bn);
  k.n = k.na + udiv(hi - k.wrap + bn - 1, bn);
  return k;
}
// First key position of tile t and how many of its bn positions exist (the rest is masked).
__host__ __device__ inline void key_tile(const KeyTiles& k, int64_t t, int bn, int64_t* j0, int* valid) {
  int64_t end;
  if (t < k.na) {
    *j0 = k.lo + t * bn;
    end = k.wrap;
  } else {
    *j0 = k.wrap + (t - k.na) * bn;
    end = k.hi;
  }
  const int64_t v = end - *j0;
  *valid = (int)(v < bn ? v : bn);
}

// Line cost of a key tile, and of the lead placeholders ahead of a unit's tiles (the cost of
// starting a piece: operand loads, pipeline fill, the epilogue).  A split-K tile of a unit
// with more than 16 rows (two MMA row groups per warp) costs about 1.5x one of at most 16
// rows, and a piece 4-6 small tiles (a least-squares fit of the split-K CTAs' finishing times
// on their tile counts by row class and their piece counts, on decode and mixed steps: 0.6-0.8
// us per small tile, 1.0-1.1 us per large one, 3.2 us per piece of 8-row units, 4-4.9 us on
// the mixed steps), so the split-K route's line counts 4 and 6 units per tile and 20 units
// of lead (leads of 16 or 24 by rows measured no better).  Prefill tiles cost 1 and a prefill
// piece 6 (about 4 us against 0.7 us per 128-key tile).
__host__ __device__ __forceinline__ int64_t tile_cost(int route, int rows) {
  return route == kRouteSplitk ? (rows > 16 ? 6 : 4) : 1;
}
__host__ __device__ __forceinline__ int64_t lead_cost(int route) { return route == kRouteSplitk ? 20 : 6; }
// CTAs that share a phase of Wp line units: at most one per costliest tile, so that every
// CTA's share holds the start of a tile of each unit it crosses (nslots stays exact).
__host__ __device__ __forceinline__ int64_t phase_ctas(int64_t G, int64_t Wp, int route) {
  const int64_t g = Wp / (route == kRouteSplitk ? 6 : 1);
  return g < 1 ? 1 : (g < G ? g : G);
}
// The tiles [ta, tb) of a unit whose first tile starts at line position k0 (nt tiles of tw
// units each) that a share [t0, t1) owns: those whose start lies in the share.
__host__ __device__ inline void line_tiles(int64_t t0, int64_t t1, int64_t k0, int64_t nt, int64_t tw,
                                           int64_t* ta, int64_t* tb) {
  const int64_t a = t0 > k0 ? t0 - k0 : 0, e = nt * tw, b = t1 - k0 < e ? t1 - k0 : e;
  *ta = (a + tw - 1) / tw;
  *tb = b > 0 ? (b + tw - 1) / tw : 0;
  if (*ta > nt) *ta = nt;
}

// Stream-K partition: CTA g of G owns flattened tiles [g*W/G, (g+1)*W/G).
__host__ __device__ inline int64_t sk_start(int64_t g, int64_t W, int64_t G) { return udiv(g * W, G); }
// CTA whose range holds tile x.
__host__ __device__ inline int64_t sk_owner(int64_t x, int64_t W, int64_t G) {
  return udiv((x + 1) * G - 1, W);
}

// All loads here are independent, so they travel together: the header, phase 0's bounds
// and this CTA's entry in phase 0 (read with the launched grid, which is the grid the
// scheduler planned for; the entry is only used if the CTA works in phase 0).
__device__ inline void walk_begin(PieceWalk& w, const Workspace& W, int route) {
  const SchedHdr* h = W.hdr;
  w.W = &W;
  w.route = route;
  w.G = gridDim.x;
  w.nphase = h->nphase[route];
  w.U = h->units[route];
  w.pb0 = h->phase_base[route][0];
  w.pb1 = h->phase_base[route][1];
  w.fu0 = W.first_unit[route][blockIdx.x];
  w.amask = h->aligned[route];
  w.p = -1;
  w.t0 = w.t1 = 0;
  w.u = 0;
}

// Moves to the next phase in which this CTA owns tiles; false when there is none.
__device__ inline bool walk_phase(PieceWalk& w) {
  const SchedHdr* h = w.W->hdr;
  while (++w.p < w.nphase) {
    const int64_t b0 = w.p == 0 ? w.pb0 : h->phase_base[w.route][w.p];
    const int64_t Wp = (w.p == 0 ? w.pb1 : h->phase_base[w.route][w.p + 1]) - b0;
    if (Wp <= 0) continue;
    if ((w.amask >> w.p) & 1) {
      // one whole unit per CTA: its span, and the walk starts at it
      const int64_t u = h->phase_unit0[w.route][w.p] + blockIdx.x;
      if (u >= h->phase_unit0[w.route][w.p + 1]) continue;
      const UnitRec& r = w.W->units[w.route][u];
      if (r.ntiles == 0) continue;
      w.t0 = r.tile_base;
      w.t1 = r.tile_base + lead_cost(w.route) + (int64_t)r.ntiles * tile_cost(w.route, r.rows);
      w.u = u;
      return true;
    }
    const int64_t Gp = phase_ctas(w.G, Wp, w.route);
    if ((int64_t)blockIdx.x >= Gp) continue;
    w.t0 = b0 + sk_start(blockIdx.x, Wp, Gp);
    w.t1 = b0 + sk_start(blockIdx.x + 1, Wp, Gp);
    if (w.t0 >= w.t1) continue;
    // the unit whose span holds tile t0, recorded by the scheduler
    w.u = w.p == 0 ? w.fu0 : w.W->first_unit[w.route][w.p * w.G + blockIdx.x];
    return true;
  }
  return false;
}

// Next piece of this CTA: a unit and its tiles [ta, tb) that this CTA processes.
__device__ inline bool walk_next(PieceWalk& w, UnitRec& ur, int64_t& ta, int64_t& tb) {
  for (;;) {
    while (w.t0 < w.t1 && w.u < w.U) {
      const UnitRec r = w.W->units[w.route][w.u];
      const int64_t tw = tile_cost(w.route, r.rows);
      const int64_t k0 = r.tile_base + lead_cost(w.route), k1 = k0 + r.ntiles * tw;  // its key tiles
      if (r.ntiles == 0 || w.t0 >= k1) {
        ++w.u;
        continue;
      }
      line_tiles(w.t0, w.t1, k0, r.ntiles, tw, &ta, &tb);
      if (ta >= tb) {
        if (w.t1 <= k1) {  // the share ends before the unit's next tile starts
          w.t0 = w.t1;
          break;
        }
        ++w.u;  // the share starts past the unit's last tile start
        continue;
      }
      ur = r;
      w.t0 = k0 + tb * tw;
      ++w.u;
      return true;
    }
    if (!walk_phase(w)) return false;
  }
}

// ------------------------------------------------------------------------------------
// inline PTX helpers
// ------------------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream serialisation
// may start while the previous kernel of the stream drains; it must wait here before reading
// anything that kernel (or an earlier one) wrote.  Without that launch attribute the wait
// returns at once.  launch_dependents lets the next such kernel start launching.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" :::); }

// A count that one kernel publishes and a concurrently running one waits for: a CTA's writes
// before a barrier, then one thread's release add, are visible to a reader whose acquire load
// sees the add.  (The callers put a barrier right before the add, which also keeps the
// compiler from moving the CTA's writes past it.)
__device__ __forceinline__ void red_add_release(int32_t* p, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;\n" ::"l"(p), "r"(v));
}
__device__ __forceinline__ int32_t ld_acquire(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool pred) {
  int sz = pred ? 16 : 0;  // src-size 0 fills the 16 bytes with zeros
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
// The same, hinting the L2 to fetch the whole 256-byte block around `src` from DRAM: the
// CTA's other threads read the rest of that store row in the same instruction.
__device__ __forceinline__ void cp_async_16_row(uint32_t dst, const void* src, bool pred) {
  int sz = pred ? 16 : 0;
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 f32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// 2^x on the SFU (PTX ex2.approx; -inf gives +0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Swizzled offset (bytes) of 16-byte chunk `c` of row `r` in a tile whose rows are
// `row_bytes` long: the low three bits of the chunk index are XORed with the row, so
// eight consecutive rows at one logical chunk hit eight different bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
  return (uint32_t)(r * row_bytes + ((c ^ (r & 7)) << 4));
}

}  // namespace sdpa
