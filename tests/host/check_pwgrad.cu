// CPU check of pwgrad_kernel's shared-memory and workspace indexing for the planner's plans.
#include <cstdio>
#include <cstdlib>
#include "large_pwgrad.cuh"

using namespace dwconv;
using namespace dwconv::large;
static int fails = 0;

template <int K>
void check(const Conv& c) {
  using Gm = PWGeo<K>;
  PWCfg g;
  size_t smem = 0;
  if (!plan_pwgrad<K>(c, &g, &smem)) {
    printf("K=%d H=%lld W=%lld: no plan\n", K, (long long)c.H, (long long)c.W);
    return;
  }
  bool ok = smem <= 227 * 1024 && smem == (size_t)g.stages * g.stage_elems * 8 && g.xrs % 2 == 0 &&
            g.grs % 2 == 0 && g.x_elems == g.xrows * g.xrs && g.gcols % 2 == 0 && g.gcols >= c.Wo &&
            g.grs >= g.gcols && (int64_t)g.x_elems + (int64_t)g.bo * g.grs <= g.stage_elems &&
            (int64_t)Gm::G * K * K + 8 <= 2LL * g.stage_elems && g.bands * g.bo >= c.Ho &&
            (g.bands - 1) * g.bo < c.Ho && Gm::threads <= 256;
  // staging writes
  for (int rr = 0; rr < g.xrows && ok; ++rr)
    for (int col = 0; col < g.xcols; ++col)
      if (rr * g.xrs + col >= g.x_elems || col >= g.xrs) { ok = false; break; }
  // reads
  const int nst = g.gcols / 2;
  for (int band = 0; band < g.bands && ok; ++band) {
    const int oh0 = band * g.bo, rows = (int)c.Ho - oh0 < g.bo ? (int)c.Ho - oh0 : g.bo;
    for (int t = 0; t < Gm::threads && ok; ++t) {
      int ib, grp, ia;
      Gm::split(t, ib, grp, ia);
      if (ia >= Gm::NA) continue;
      if (ib >= Gm::NB || grp >= Gm::G) { ok = false; break; }
      const int a0 = Gm::RA * ia, b0 = 8 * ib;
      int lo = g.pad - oh0 - a0 - (Gm::RA - 1), hi = g.pad + (int)c.H - oh0 - a0;
      lo = lo < 0 ? 0 : lo;
      hi = hi > rows ? rows : hi;
      for (int oh = grp; oh < hi; oh += Gm::G) {
        if (oh < lo) continue;
        for (int ra = 0; ra < Gm::RA; ++ra) {
          const int row = oh + a0 + ra;
          if (row >= g.xrows) { ok = false; break; }
          for (int m = 0; m <= nst + 3; ++m) {
            const int q = b0 + 2 * m;
            if (q + 1 >= g.xcols || q + 1 >= g.xrs || q % 2) { ok = false; break; }
          }
        }
        if (oh * g.grs + 2 * (nst - 1) + 1 >= g.bo * g.grs) ok = false;
      }
      // every tap the thread writes back is in range
    }
  }
  // every (ib, grp, ia) appears exactly once among the threads
  {
    static int seen[64][256][64];
    for (int a = 0; a < Gm::NB; ++a) for (int b = 0; b < Gm::G; ++b) for (int d = 0; d < Gm::NA; ++d) seen[a][b][d] = 0;
    for (int t = 0; t < Gm::threads; ++t) {
      int ib, grp, ia;
      Gm::split(t, ib, grp, ia);
      if (ia < Gm::NA) seen[ib][grp][ia]++;
    }
    for (int a = 0; a < Gm::NB; ++a) for (int b = 0; b < Gm::G; ++b) for (int d = 0; d < Gm::NA; ++d) if (seen[a][b][d] != 1) ok = false;
  }
  // the tap blocks cover the filter
  if (Gm::NA * Gm::RA < K || Gm::NB * 8 < K) ok = false;
  // sample chunks: whole pairs (an even count), covering the batch exactly
  if (c.N >= 1 && (g.nb % 2 || (int64_t)g.chunks * g.nb < c.N || (int64_t)(g.chunks - 1) * g.nb >= c.N)) ok = false;
  if (!ok) ++fails;
  printf("%s K=%2d N=%lld C=%lld H=%3lld W=%3lld p=%2d: chunks=%d bands=%d bo=%d xrows=%d xrs=%d grs=%d stages=%d "
         "smem=%zu KB thr=%d G=%d conf=%d\n",
         ok ? "ok  " : "FAIL", K, (long long)c.N, (long long)c.C, (long long)c.H, (long long)c.W, g.pad, g.chunks,
         g.bands, g.bo, g.xrows, g.xrs, g.grs, g.stages, smem / 1024, Gm::threads, Gm::G,
         pw_conflicts<K>(g, Gm::threads));
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
  for (int h : {7, 9, 16, 23, 32, 33, 48, 57, 64, 96, 111, 112, 128})
    for (int p : {K / 2, 0, K - 1})
      for (long n : {1L, 3L, 16L, 64L}) {
        Conv c = mk(n, 5, h, h + (h % 3), K, p);
        if (c.Ho < 1 || c.Wo < 1 || c.Ho > 128 || c.Wo > 128) continue;
        check<K>(c);
      }
}

int main() {
  sweep<7>(); sweep<9>(); sweep<13>(); sweep<21>(); sweep<27>(); sweep<29>(); sweep<31>();
  for (int h : {32, 48, 64})
    for (int k : {13, 21, 27, 31}) {
      if (k == 13) check<13>(mk(64, 384, h, h, 13, 6));
      if (k == 21) check<21>(mk(64, 384, h, h, 21, 10));
      if (k == 27) check<27>(mk(64, 384, h, h, 27, 13));
      if (k == 31) check<31>(mk(64, 384, h, h, 31, 15));
    }
  printf("fails: %d\n", fails);
  return fails != 0;
}
