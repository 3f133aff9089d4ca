// CPU check of the tensor-core forward / grad-input's index arithmetic: the
// tensor- and shared-memory plan, the K steps each tile visits (every input
// position a tile's outputs reach must be inside them), and the builders'
// A operand -- each 8-tap piece loaded from the eight shifted copies of the
// padded filter -- replayed for every tile and checked against a direct
// integer correlation.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "ibgemm.cu"

using namespace dwconv;
using namespace dwconv::ibg;
static int fails = 0, cases = 0, walked = 0;

Conv mk(long N, long C, long H, long W, int kh, int kw, int ph, int pw) {
  Conv c{};
  c.N = N; c.C = C; c.H = H; c.W = W; c.m = 1; c.kh = kh; c.kw = kw; c.sh = c.sw = 1; c.ph = ph; c.pw = pw;
  c.dh = c.dw = 1; c.Ho = H + 2 * ph - (kh - 1); c.Wo = W + 2 * pw - (kw - 1); c.off = 0; c.ctot = C;
  c.dtype = DWCONV_F16;
  return c;
}

void check(const Conv& c, bool flip) {
  if (c.Ho < 1 || c.Wo < 1 || !geo_supported(c, flip)) return;
  ++cases;
  bool ok = true;
  const Geo q = geo_of(c, flip);
  ICfg g{};
  g.Hi = q.Hi; g.Wi = q.Wi; g.Ho = q.Ho; g.Wo = q.Wo;
  g.kh = c.kh; g.kw = c.kw; g.ph = q.ph; g.pw = q.pw;
  g.flip = flip;
  g.T = (g.Ho * g.Wo + kM - 1) / kM;
  g.L = row_len(g.Wi, g.Wo);
  g.nb = tile::round_up((int)c.N, 16);
  // the launch's tensor-memory layout: accumulators, then the A stages
  g.acc_cols = tile::round_up(g.nb, 32);
  g.nacc = 2 * g.acc_cols + 32 * kAtoms * kS <= 512 ? 2 : 1;
  g.acol = g.nacc * g.acc_cols;
  g.ncols = 32;
  while (g.ncols < g.acol + 32 * kAtoms * kS) g.ncols *= 2;
  if (g.ncols > 512 || g.nb > 256 || g.nb < 16) ok = false;
  if (smem_bytes(kS * kAtoms, g.nb, g.kh, g.L) > 227 * 1024) ok = false;
  // padded rows: 16-byte pieces, the eight copies in different bank groups
  if (g.L % 8 || (g.L / 8) % 2 == 0 || g.L < g.Wo + g.Wi - 1 + 8 || g.Wi % 8) ok = false;

  const int kh = g.kh, kw = g.kw, HW = g.Hi * g.Wi, F = g.Ho * g.Wo;
  std::vector<int> w(kh * kw), x(HW);
  for (auto& v : w) v = rand() % 7 - 3;
  for (auto& v : x) v = rand() % 7 - 3;
  // the correlation's filter (stored filter rotated for the grad-input)
  auto wcorr = [&](int dy, int dx) { return flip ? w[(kh - 1 - dy) * kw + (kw - 1 - dx)] : w[dy * kw + dx]; };
  // K-step coverage: every input position a tile's outputs read
  for (int t = 0; t < g.T && ok; ++t) {
    int lo, hi;
    k_range(g, t, lo, hi);
    if (lo < 0 || hi > (HW + kKs - 1) / kKs || lo >= hi) { ok = false; break; }
    for (int f = t * kM; f < t * kM + kM && f < F; ++f) {
      const int oh = f / g.Wo, ow = f % g.Wo;
      for (int dy = 0; dy < kh; ++dy) {
        const int ih = oh - g.ph + dy;
        if (ih < 0 || ih >= g.Hi) continue;
        for (int dx = 0; dx < kw; ++dx) {
          const int iw = ow - g.pw + dx;
          if (iw < 0 || iw >= g.Wi) continue;
          const int kc = (ih * g.Wi + iw) / kKs;
          if (kc < lo || kc >= hi) ok = false;
        }
      }
    }
  }
  // the builders' A operand and the GEMM it feeds, on planes small enough to walk
  if (ok && (long)F * HW <= (1L << 22)) {
    ++walked;
    // SC[s][dy][i] = filter row dy at column i + s - (Wo - 1 - pw), zero outside
    std::vector<int> sc((size_t)8 * kh * g.L);
    for (int s = 0; s < 8; ++s)
      for (int dy = 0; dy < kh; ++dy)
        for (int i = 0; i < g.L; ++i) {
          const int b = i + s - (g.Wo - 1 - g.pw);
          sc[((size_t)s * kh + dy) * g.L + i] = (b >= 0 && b < kw) ? wcorr(dy, b) : 0;
        }
    for (int t = 0; t < g.T && ok; ++t) {
      int lo, hi;
      k_range(g, t, lo, hi);
      for (int m = 0; m < kM; ++m) {
        const int f = t * kM + m;
        if (f >= F) break;
        const int oh = f / g.Wo, ow = f % g.Wo, j0 = g.Wo - 1 - ow;
        long y = 0, ref = 0;
        for (int kc = lo; kc < hi; ++kc)
          for (int half = 0; half < kAtoms; ++half)
            for (int j = 0; j < 8; ++j) {
              const int p0 = kc * kKs + kAtom * half + 8 * j;  // first position of the piece
              const int ih = p0 / g.Wi, iw = p0 % g.Wi;
              const int dy = ih - oh + g.ph;
              if (dy < 0 || dy >= kh) continue;
              const int base = (j0 & ~7) + iw;  // element offset of the 16-byte load in its row
              if (base % 8 || base + 8 > g.L) { ok = false; continue; }
              for (int e = 0; e < 8; ++e) {
                if (p0 + e >= HW) continue;  // past the plane: zero-filled B rows
                y += (long)sc[((size_t)(j0 & 7) * kh + dy) * g.L + base + e] * x[p0 + e];
              }
            }
        for (int dy = 0; dy < kh; ++dy)
          for (int dx = 0; dx < kw; ++dx) {
            const int ih = oh - g.ph + dy, iw = ow - g.pw + dx;
            if (ih >= 0 && ih < g.Hi && iw >= 0 && iw < g.Wi) ref += (long)wcorr(dy, dx) * x[ih * g.Wi + iw];
          }
        if (y != ref) { ok = false; break; }
      }
    }
  }
  if (!ok) {
    ++fails;
    printf("FAIL N=%lld H=%lld W=%lld k=%dx%d p=%d,%d flip=%d\n", (long long)c.N, (long long)c.H, (long long)c.W,
           kh, kw, c.ph, c.pw, (int)flip);
  }
}

int main() {
  srand(2);
  for (int W : {8, 16, 24, 32, 40, 48, 64, 96, 128})
    for (int H : {1, 5, 8, 17, 32, 33, 64, 100, 128})
      for (int k : {9, 13, 17, 21, 27, 31})
        for (int phs : {0, 1, 2})
          for (long N : {1L, 64L, 256L}) {
            const int p = phs == 0 ? k / 2 : phs == 1 ? 0 : k - 1;
            for (bool flip : {false, true}) check(mk(N, 3, H, W, k, k, p, p), flip);
          }
  // non-square filters and mixed padding
  for (int W : {16, 32, 64})
    for (int H : {9, 32, 48})
      for (int kh : {9, 15, 31})
        for (int kw : {9, 21, 31})
          for (bool flip : {false, true}) check(mk(16, 2, H, W, kh, kw, kh / 2, kw - 1), flip);
  printf("cases %d walked %d fails %d\n", cases, walked, fails);
  return fails != 0 || cases == 0;
}
