// CPU check of pconv_kernel's shared-memory indexing for the planner's plans.
#include <cstdio>
#include <cstdlib>
#include "large_pair.cuh"

using namespace dwconv;
using namespace dwconv::large;

static int fails = 0;

template <int K, int V>
void check_plan(const Conv& c, bool flip, int fbo = 0, int fppu = 0, int fst = 0) {
  PCfg g;
  int threads = 0;
  double score = 0;
  if (!plan_pair<K, V>(c, flip, &g, &threads, &score, fbo, fppu, fst)) {
    if (!fbo && !fppu && !fst) printf("K=%d V=%d H=%lld W=%lld: no plan\n", K, V, (long long)c.H, (long long)c.W);
    return;
  }
  constexpr int KP2 = FiltGeo<K>::KP2;
  constexpr int NWP = V + K - 1, NCH = NWP / 2;
  const long smem = (long)g.stages * g.stage_elems * 8;
  bool ok = smem <= 227 * 1024 && g.stage_elems == g.ppu * g.blk && (g.blk % 2) == 0 && (g.rs % 2) == 0 &&
            threads >= 32 && threads <= 288 && threads % 32 == 0;
  // staging writes (pairs) of the tile and of the filter table
  for (int pp = 0; pp < g.ppu && ok; ++pp)
    for (int r = 0; r < g.tr && ok; ++r)
      for (int col = 0; col < g.cols; ++col) {
        const long o = (long)pp * g.blk + (long)r * g.rs + pphys<V>(col);
        if (o < (long)pp * g.blk || o >= (long)pp * g.blk + g.fofs || pphys<V>(col) >= g.rs) { ok = false; break; }
      }
  for (int pp = 0; pp < g.ppu && ok; ++pp)
    for (int a = 0; a < K; ++a)
      for (int b = 0; b < KP2; ++b) {
        const long o = (long)pp * g.blk + g.fofs + a * KP2 + b;
        if (o >= (long)(pp + 1) * g.blk) { ok = false; break; }
      }
  // reads of every item of every band
  for (int band = 0; band < g.nbands && ok; ++band) {
    const int rows = (g.Hout - band * g.bo) < g.bo ? (g.Hout - band * g.bo) : g.bo;
    for (int it = 0; it < g.items && ok; ++it) {
      const int cbi = it % g.cb, slot0 = it / g.cb, pp = slot0 % g.ppu, slot = slot0 / g.ppu;
      if (slot >= rows) continue;
      const int ohr = slot_row(slot, rows, g.mirror);
      if (ohr < 0 || ohr >= rows) { ok = false; break; }
      const int oh = band * g.bo + ohr;
      int a_lo = g.pad - oh; a_lo = a_lo < 0 ? 0 : a_lo;
      int a_hi = g.Hin + g.pad - oh; a_hi = a_hi > K ? K : a_hi;
      for (int a = a_lo; a < a_hi; ++a) {
        if (ohr + a >= g.tr) { ok = false; break; }
        const long xb = (long)pp * g.blk + (long)(ohr + a) * g.rs + (V + 2) * cbi;
        for (int s = 0; s < NCH; ++s) {
          const long o = xb + 2 * (s + s / (V / 2));
          if (o % 2 || o + 1 >= (long)pp * g.blk + (long)(ohr + a + 1) * g.rs) { ok = false; break; }
          // logical columns of this chunk must be staged
          const int lcol = V * cbi + 2 * s + 1;
          if (lcol >= g.cols) { ok = false; break; }
          // the input column it stands for, relative to the output column
        }
        const long fb = (long)pp * g.blk + g.fofs + (long)a * KP2;
        for (int b = 0; b < K; b += 2)
          if (fb + b + 1 >= (long)(pp + 1) * g.blk || (fb + b) % 2) { ok = false; break; }
      }
    }
    // every output row of the band covered exactly once
    int* seen = (int*)calloc(rows > 0 ? rows : 1, sizeof(int));
    for (int s = 0; s < rows; ++s) seen[slot_row(s, rows, g.mirror)]++;
    for (int r = 0; r < rows; ++r) if (seen[r] != 1) ok = false;
    free(seen);
  }
  if (!ok) ++fails;
  printf("%s K=%2d V=%2d %s N*C=%lld H=%3lld W=%3lld pad=%2d: bo=%d nb=%d ppu=%d thr=%d stages=%d smem=%ld KB "
         "rs=%d blk=%d units=%lld score=%.3f conf=%d\n",
         ok ? "ok  " : "FAIL", K, V, flip ? "bwd" : "fwd", (long long)(c.N * c.C), (long long)c.H, (long long)c.W,
         g.pad, g.bo, g.nbands, g.ppu, threads, g.stages, smem / 1024, g.rs, g.blk, (long long)g.units, score,
         pair_conflicts<K, V>(g, threads));
}

Conv mk(long N, long C, long H, long W, int k, int p) {
  Conv c{};
  c.N = N; c.C = C; c.H = H; c.W = W; c.m = 1; c.kh = c.kw = k; c.sh = c.sw = 1; c.ph = c.pw = p; c.dh = c.dw = 1;
  c.Ho = H + 2 * p - (k - 1); c.Wo = W + 2 * p - (k - 1);
  c.off = 0; c.ctot = C; c.dtype = 0;
  c.dC = FastDiv((uint32_t)C);
  return c;
}

template <int K>
void sweep() {
  const int hs[] = {7, 8, 13, 16, 24, 28, 32, 33, 40, 48, 56, 63, 64, 96, 100, 128};
  for (int h : hs)
    for (int p : {K / 2, 0, K - 1}) {
      Conv c = mk(3, 5, h, h + (h % 3), K, p);
      if (c.Ho < 1 || c.Wo < 1) continue;
      check_plan<K, 16>(c, false);
      check_plan<K, 8>(c, false);
      check_plan<K, 16>(c, true);
    }
}

int main() {
  sweep<7>(); sweep<13>(); sweep<21>(); sweep<27>(); sweep<31>(); sweep<9>(); sweep<29>();
  for (int h : {32, 48, 64}) {
    check_plan<31, 16>(mk(64, 384, h, h, 31, 15), false);
    check_plan<31, 8>(mk(64, 384, h, h, 31, 15), false);
    check_plan<13, 16>(mk(64, 384, h, h, 13, 6), false);
    check_plan<21, 16>(mk(64, 384, h, h, 21, 10), false);
    check_plan<27, 16>(mk(64, 384, h, h, 27, 13), false);
  }
  for (int h : {32, 48, 64})
    for (int bo : {0, h, h / 2, h / 4})
      for (int ppu : {0, 1, 2, 3, 4})
        for (int st : {1, 2}) {
          check_plan<31, 16>(mk(64, 384, h, h, 31, 15), false, bo, ppu, st);
          check_plan<31, 8>(mk(64, 384, h, h, 31, 15), false, bo, ppu, st);
          check_plan<13, 16>(mk(64, 384, h, h, 13, 6), false, bo, ppu, st);
          check_plan<13, 8>(mk(64, 384, h, h, 13, 6), false, bo, ppu, st);
          check_plan<21, 16>(mk(64, 384, h, h, 21, 10), true, bo, ppu, st);
          check_plan<27, 8>(mk(64, 384, h, h, 27, 13), false, bo, ppu, st);
        }
  printf("fails: %d\n", fails);
  return fails != 0;
}
