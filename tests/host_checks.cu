// Host-side checks of the arithmetic the kernels share with the host (built with nvcc as a
// host program, run by tests/test_host_arith.py):
//   * udiv against plain 64-bit division, operands above 2^32 included;
//   * the stream-K partition: shares are contiguous, cover [0, W) once, and sk_owner(x)
//     names the CTA whose share holds x;
//   * the cost-weighted tile line: each tile owned once, a unit's owners consecutive, each
//     owning a tile;
//   * the small scheduler's admission bound on the units of any live table;
//   * the key tiles of a prefill unit: they cover its keys once and never wrap a ring;
//   * the workspace layout: every region 256-byte aligned, disjoint, inside the size it
//     returns, and the partial slots sized for the phases the scheduler may use;
//   * segment_bits for a grid of segments, printed one per line for comparison with the
//     oracle's own rule.
#include <cstdio>
#include <cstdlib>
#include <vector>
#include <algorithm>

#include "../varlen_gqa_attention_gb300/csrc/common.cuh"

using namespace sdpa;

static int failures = 0;
#define CHECK(c)                                                              \
  do {                                                                        \
    if (!(c)) {                                                               \
      std::printf("FAIL %s:%d %s\n", __FILE__, __LINE__, #c);                 \
      ++failures;                                                             \
    }                                                                         \
  } while (0)

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64() {  // xorshift64*
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return rng_state * 0x2545F4914F6CDD1Dull;
}

int main() {
  // udiv
  for (int i = 0; i < 200000; ++i) {
    const int64_t a = (int64_t)(next_u64() >> (1 + next_u64() % 40));
    const int64_t b = (int64_t)(next_u64() >> (1 + next_u64() % 60)) + 1;
    CHECK(udiv(a, b) == a / b);
  }
  // stream-K partition
  for (int i = 0; i < 20000; ++i) {
    const int64_t W = 1 + (int64_t)(next_u64() % 100000);
    const int64_t G = 1 + (int64_t)(next_u64() % std::min<int64_t>(W, 2000));
    int64_t prev_end = 0;
    for (int64_t g = 0; g < G; ++g) {
      const int64_t a = sk_start(g, W, G), b = sk_start(g + 1, W, G);
      CHECK(a == prev_end && b > a);
      CHECK(sk_owner(a, W, G) == g && sk_owner(b - 1, W, G) == g);
      prev_end = b;
    }
    CHECK(prev_end == W);
  }
  // the cost-weighted tile line of one phase: units of nt tiles of tile_cost units each,
  // behind lead_cost placeholders, shared by phase_ctas CTAs.  Every tile is owned by exactly
  // one CTA (the one whose share holds its start, line_tiles), the owners of a unit's tiles
  // are the CTAs from sk_owner(first start) to sk_owner(last start), and each of them owns
  // at least one of its tiles (so a unit's slot count is exact)
  for (int i = 0; i < 3000; ++i) {
    const int route = (next_u64() & 1) ? kRouteSplitk : kRoutePrefill;
    const int nu = 1 + (int)(next_u64() % 40);
    std::vector<int64_t> base(nu), nts(nu), tws(nu), lds(nu);
    int64_t Wp = 0;
    for (int u = 0; u < nu; ++u) {
      nts[u] = (next_u64() % 5 == 0) ? 0 : 1 + (int64_t)(next_u64() % ((next_u64() & 1) ? 4 : 300));
      const int rows = 1 + (int)(next_u64() % 32);
      tws[u] = tile_cost(route, rows);
      lds[u] = lead_cost(route);
      base[u] = Wp;
      Wp += nts[u] > 0 ? lds[u] + nts[u] * tws[u] : 0;
    }
    if (Wp == 0) continue;
    const int64_t G = 1 + (int64_t)(next_u64() % 400);
    const int64_t Gp = phase_ctas(G, Wp, route);
    CHECK(Gp >= 1 && Gp <= G);
    for (int u = 0; u < nu; ++u) {
      if (nts[u] == 0) continue;
      const int64_t k0 = base[u] + lds[u];
      std::vector<int> owner(nts[u], -1);
      for (int64_t g = 0; g < Gp; ++g) {
        int64_t ta, tb;
        line_tiles(sk_start(g, Wp, Gp), sk_start(g + 1, Wp, Gp), k0, nts[u], tws[u], &ta, &tb);
        for (int64_t t = ta; t < tb; ++t) {
          CHECK(owner[t] == -1);
          owner[t] = (int)g;
        }
      }
      const int64_t g0 = sk_owner(k0, Wp, Gp), g1 = sk_owner(k0 + (nts[u] - 1) * tws[u], Wp, Gp);
      CHECK(owner[0] == g0 && owner[nts[u] - 1] == g1);
      for (int64_t t = 0; t < nts[u]; ++t) {
        CHECK(owner[t] >= 0);
        if (t > 0) CHECK(owner[t] == owner[t - 1] || owner[t] == owner[t - 1] + 1);
      }
    }
  }
  // the small scheduler's admission bound: for every call sched_small_ok admits, any table
  // of disjoint live segments, routed any way, gives at most kSchedThreads threads of units
  // with route 2's starting at a warp boundary
  for (int i = 0; i < 20000; ++i) {
    const int Hkv = 1 << (int)(next_u64() % 4);
    const int group = 1 + (int)(next_u64() % 16);
    const int Hq = Hkv * group;
    const int S = 1 + (int)(next_u64() % 40);
    const int64_t T = 1 + (int64_t)(next_u64() % ((next_u64() & 1) ? 300 : 9000));
    if (!sched_small_ok(T, Hq, Hkv, S)) continue;
    CHECK(S <= kSmallSegs && T <= 8192);
    int64_t left = T, u1 = 0, u2 = 0;
    for (int s = 0; s < S && left > 0; ++s) {
      const int64_t ql = 1 + (int64_t)(next_u64() % (uint64_t)left);
      left -= ql;
      const int64_t R = ql * group;
      if (next_u64() & 1) u1 += Hkv * ((R + kSplitkRows - 1) / kSplitkRows);
      else {
        const int rpu = prefill_unit_rows(64 << (int)(next_u64() % 3));
        u2 += Hkv * ((R + rpu - 1) / rpu);
      }
    }
    CHECK(((u1 + 31) / 32) * 32 + u2 <= kSchedThreads);
    // the table that comes closest to the bound: S - 1 one-row segments and one long one, all
    // on the split-K route but the first, on the prefill route (route 2 after padding)
    if (T >= S) {
      int64_t w1 = 0;
      for (int s = 1; s < S - 1; ++s) w1 += Hkv * ((group + kSplitkRows - 1) / kSplitkRows);
      if (S > 1) w1 += Hkv * (((T - S + 1) * group + kSplitkRows - 1) / kSplitkRows);
      const int64_t w2 = S > 1 ? Hkv * ((group + 255) / 256) : 0;
      CHECK(((w1 + 31) / 32) * 32 + w2 <= kSchedThreads);
    }
  }
  // key tiles of a prefill unit: the tiles cover [lo, hi) once, in order, each 1..bn keys,
  // and no tile's store rows wrap (its first and last key sit in one block of `rows`)
  for (int i = 0; i < 200000; ++i) {
    const int64_t rows = 1 + (int64_t)(next_u64() % 5000);
    const int bn = (next_u64() & 1) ? 128 : 64;
    const int64_t lo = (int64_t)(next_u64() % 100000);
    const int64_t span = (int64_t)(next_u64() % (rows + 1));  // a unit's keys span <= rows
    const int64_t hi = lo + span;
    const KeyTiles kt = key_tiles(lo, hi, rows, bn);
    int64_t expect = lo;
    for (int64_t t = 0; t < kt.n; ++t) {
      int64_t j0;
      int valid;
      key_tile(kt, t, bn, &j0, &valid);
      CHECK(j0 == expect && valid >= 1 && valid <= bn);
      CHECK(j0 / rows == (j0 + valid - 1) / rows);
      expect = j0 + valid;
    }
    CHECK(expect == (span > 0 ? hi : lo));
    CHECK(kt.n <= (span + bn - 1) / bn + 1);
  }
  // workspace layout
  const int64_t Ts[] = {1, 32, 513, 4096, 100000};
  const int Ss[] = {1, 7, 32, 1500};
  const int Ds[] = {64, 128, 256};
  for (int64_t T : Ts)
    for (int S : Ss)
      for (int D : Ds) {
        const int Hq = 16, Hkv = 2;
        const int64_t gs = 304, gp = 152;
        Workspace ws{};
        const size_t need = layout_workspace(nullptr, T, Hq, Hkv, D, S, gs, gp, nullptr);
        char* base = (char*)(uintptr_t)4096;  // addresses only, never dereferenced
        const size_t need2 = layout_workspace(base, T, Hq, Hkv, D, S, gs, gp, &ws);
        CHECK(need == need2);
        struct R {
          const void* p;
          int64_t bytes;
        };
        std::vector<R> rs = {{ws.hdr, (int64_t)sizeof(SchedHdr)},
                             {ws.segs, (int64_t)sizeof(SegRec) * S},
                             {ws.row_seg, 4 * T},
                             {ws.row_info, 16 * T},
                             {ws.seg_flag, 4 * (int64_t)S}};
        const int64_t grid[3] = {0, gs, gp};
        const int rpu[3] = {0, kSplitkRows, prefill_unit_rows(D)};
        for (int r = 1; r < 3; ++r) {
          CHECK(ws.unit_cap[r] == unit_cap(T, Hq, Hkv, S, rpu[r]));
          CHECK(ws.part_cap[r] >= (ws.unit_cap[r] + (int64_t)kPartPhases * grid[r] + 1) * rpu[r]);
          rs.push_back({ws.units[r], (int64_t)sizeof(UnitRec) * ws.unit_cap[r]});
          rs.push_back({ws.first_unit[r], 4 * (int64_t)kMaxPhases * grid[r]});
          rs.push_back({ws.part_ml[r], 8 * ws.part_cap[r]});
          rs.push_back({ws.part_o[r], 4 * ws.part_cap[r] * D});
        }
        rs.push_back({ws.unit_done, 4 * ws.unit_cap[kRouteSplitk]});
        std::sort(rs.begin(), rs.end(), [](const R& x, const R& y) { return x.p < y.p; });
        for (size_t k = 0; k < rs.size(); ++k) {
          const uintptr_t a = (uintptr_t)rs[k].p;
          CHECK(a % 256 == 0);
          CHECK(a >= (uintptr_t)base && a + rs[k].bytes <= (uintptr_t)base + need);
          if (k + 1 < rs.size()) CHECK(a + rs[k].bytes <= (uintptr_t)rs[k + 1].p);
        }
        // every unit a route can produce fits: live segments cover disjoint rows
        CHECK(ws.unit_cap[kRouteSplitk] >= (int64_t)Hkv * ((T * (Hq / Hkv) + kSplitkRows - 1) / kSplitkRows));
      }
  // the split-K-only layout of the allocation-free entry: the same regions, the prefill
  // route's tables empty, inside the bytes it reports and no larger than the full layout
  for (int64_t T : Ts)
    for (int S : Ss)
      for (int D : Ds) {
        const int Hq = 16, Hkv = 2;
        const int64_t gs = 304;
        Workspace ws{};
        char* base = (char*)(uintptr_t)4096;
        const size_t need = layout_workspace(base, T, Hq, Hkv, D, S, gs, 0, &ws, false);
        CHECK(need == layout_workspace(nullptr, T, Hq, Hkv, D, S, gs, 0, nullptr, false));
        CHECK(need <= layout_workspace(nullptr, T, Hq, Hkv, D, S, gs, 152, nullptr, true));
        CHECK(ws.unit_cap[kRoutePrefill] == 0 && ws.part_cap[kRoutePrefill] == 0);
        CHECK(ws.unit_cap[kRouteSplitk] == unit_cap(T, Hq, Hkv, S, kSplitkRows));
        CHECK(ws.part_cap[kRouteSplitk] >= (ws.unit_cap[kRouteSplitk] + (int64_t)kPartPhases * gs + 1) * kSplitkRows);
        struct R {
          const void* p;
          int64_t bytes;
        };
        std::vector<R> rs = {{ws.hdr, (int64_t)sizeof(SchedHdr)},
                             {ws.segs, (int64_t)sizeof(SegRec) * S},
                             {ws.row_seg, 4 * T},
                             {ws.row_info, 16 * T},
                             {ws.seg_flag, 4 * (int64_t)S},
                             {ws.units[kRouteSplitk], (int64_t)sizeof(UnitRec) * ws.unit_cap[kRouteSplitk]},
                             {ws.first_unit[kRouteSplitk], 4 * (int64_t)kMaxPhases * gs},
                             {ws.part_ml[kRouteSplitk], 8 * ws.part_cap[kRouteSplitk]},
                             {ws.part_o[kRouteSplitk], 4 * ws.part_cap[kRouteSplitk] * D}};
        std::sort(rs.begin(), rs.end(), [](const R& x, const R& y) { return x.p < y.p; });
        for (size_t k = 0; k < rs.size(); ++k) {
          const uintptr_t a = (uintptr_t)rs[k].p;
          CHECK(a % 256 == 0);
          CHECK(a >= (uintptr_t)base && a + rs[k].bytes <= (uintptr_t)base + need);
          if (k + 1 < rs.size()) CHECK(a + rs[k].bytes <= (uintptr_t)rs[k + 1].p);
        }
      }
  // scratch the allocation-free entry needs for the fallback-grid test case (T=2048 packed
  // rows, Hq=16, Hkv=2, D=128, S=8) at the general grid of a 152-SM GB300 (2 split-K CTAs per
  // SM at D=128) and at one CTA per SM: "STATIC_NEED grid bytes"
  for (int64_t g : {304, 152})
    std::printf("STATIC_NEED %lld %zu\n", (long long)g,
                layout_workspace(nullptr, 2048, 16, 2, 128, 8, g, 0, nullptr, false));
  // segment_bits on a grid: "q_start q_len col kv_end T rows cols window bits"
  const int64_t vals_q[] = {-1, 0, 3};
  const int64_t lens[] = {-1, 0, 1, 5};
  const int64_t colv[] = {-1, 0, 2};
  const int64_t kvs[] = {-1, 0, 1, 6, 9, 40};
  const int wins[] = {0, -2, 1, 3};
  for (int64_t qs : vals_q)
    for (int64_t ql : lens)
      for (int64_t c : colv)
        for (int64_t ke : kvs)
          for (int w : wins)
            std::printf("SEG %lld %lld %lld %lld %d %d %d %d %d\n", (long long)qs, (long long)ql,
                        (long long)c, (long long)ke, 8, 8, 2, w,
                        segment_bits(qs, ql, c, ke, 8, 8, 2, w));
  std::printf("failures %d\n", failures);
  return failures != 0;
}
