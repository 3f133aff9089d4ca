// CPU check of the filter-cache tensor-core kernel's index arithmetic: the
// shared-memory and tensor-memory plan, the cache contents (strip taps), the
// K steps each tile visits, the strip offsets of its A operands, and the
// whole GEMM walk against a direct correlation (small integers, exact).
#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "ibgemm_cache.cu"

using namespace dwconv;
using namespace dwconv::ibc;
static int fails = 0, cases = 0;

Conv mk(long N, long C, long H, long W, int kh, int kw, int ph, int pw) {
  Conv c{};
  c.N = N; c.C = C; c.H = H; c.W = W; c.m = 1; c.kh = kh; c.kw = kw; c.sh = c.sw = 1; c.ph = ph; c.pw = pw;
  c.dh = c.dw = 1; c.Ho = H + 2 * ph - (kh - 1); c.Wo = W + 2 * pw - (kw - 1); c.off = 0; c.ctot = C;
  c.dtype = DWCONV_F16;
  return c;
}

void check(const Conv& c, bool flip) {
  Geo q;
  if (c.Ho < 1 || c.Wo < 1) return;
  if (!make_geo(c, flip, &q)) return;
  if (cache_bytes(c, flip) == 0) return;
  ++cases;
  bool ok = true;
  const int kh = c.kh, kw = c.kw;
  std::vector<int> w(kh * kw), x(q.Hi * q.Wi);
  for (auto& v : w) v = rand() % 7 - 3;
  for (auto& v : x) v = rand() % 7 - 3;
  // one channel's cache: NS strips of Wo rows x 64 taps
  const int rows = q.NS * q.Wo;
  std::vector<int> cache((size_t)rows * 64);
  for (int r = 0; r < rows; ++r)
    for (int k = 0; k < 64; ++k) {
      const int tap = strip_tap(kh, kw, q.pw, q.flip, q.Wo, q.jmax, r / q.Wo, r % q.Wo, k);
      if (tap >= kh * kw) ok = false;
      cache[(size_t)r * 64 + k] = tap >= 0 ? w[tap] : 0;
    }
  // the correlation the cached GEMM must reproduce (filter rotated for the grad-input)
  auto wf = [&](int dy, int dx) { return q.flip ? w[(kh - 1 - dy) * kw + (kw - 1 - dx)] : w[dy * kw + dx]; };
  std::vector<long> ref(q.Ho * q.Wo, 0);
  for (int oh = 0; oh < q.Ho; ++oh)
    for (int ow = 0; ow < q.Wo; ++ow) {
      long s = 0;
      for (int dy = 0; dy < kh; ++dy)
        for (int dx = 0; dx < kw; ++dx) {
          const int ih = oh - q.ph + dy, iw = ow - q.pw + dx;
          if (ih >= 0 && ih < q.Hi && iw >= 0 && iw < q.Wi) s += (long)wf(dy, dx) * x[ih * q.Wi + iw];
        }
      ref[oh * q.Wo + ow] = s;
    }
  std::vector<long> y(q.Ho * q.Wo);
  for (int nb : {16, 32, 48, 64}) {
    KCfg k{};
    size_t smem = 0;
    if (!plan_kernel(q, nb, &k, &smem)) {
      ok = false;
      printf("no plan nb=%d\n", nb);
      continue;
    }
    k.T = q.T; k.KB = q.KB; k.dmin = q.dmin; k.dmax = q.dmax;
    // shared memory: barriers (1 KB), the resident strips, B stages; every
    // block 1024-byte aligned for the 128-byte swizzle; descriptor start
    // addresses have 18 bits
    if (smem > kSmemLimit || k.stages < 2 || k.stages > kMaxStages) ok = false;
    if (k.strips_bytes % 1024 || k.stage_bytes % 1024 || k.strip_bytes != (uint32_t)q.Wo * 128) ok = false;
    if ((size_t)k.strips_bytes + 1024 + (size_t)k.stages * k.stage_bytes != smem || smem > (1u << 18)) ok = false;
    // tensor memory: nsets x G accumulators of acc_cols columns in a power-of-two allocation <= 512
    if (k.acc_cols < nb || k.acc_cols % 32 || k.nsets * k.G * k.acc_cols > k.ncols || k.ncols > 512 ||
        (k.ncols & (k.ncols - 1)) || k.ncols < 32 || k.nsets * k.G > kMaxSlots || k.nsets < 1 || k.nsets > 2)
      ok = false;
    // tile groups cover the tiles, none empty
    if (k.G * k.NG < q.T || (k.NG - 1) * k.G >= q.T || k.G < 1) ok = false;
    std::fill(y.begin(), y.end(), 0);
    for (int gi = 0; gi < k.NG; ++gi) {
      const int t0 = gi * k.G, t1 = std::min(q.T, t0 + k.G);
      int lo, hi;
      unit_range(k, t0, t1, lo, hi);
      std::vector<int> seen(q.T, 0);
      for (int kc = lo; kc < hi; ++kc) {
        // tiles of the group whose K range holds this step: t in [kc - dmax, kc - dmin]
        const int tlo = std::max(t0, kc - q.dmax), thi = std::min(t1, kc - q.dmin + 1);
        for (int t = tlo; t < thi; ++t) {
          int first, end;
          k_range(q.dmin, q.dmax, q.KB, t, first, end);
          if (kc < first || kc >= end) { ok = false; continue; }
          seen[t]++;
          for (int a = 0; a < 2; ++a) {  // the two 64-wide halves of the 128-position K step
            const int q0 = strip_of(q.jmax, q.R, q.h, q.ph, kc - t, a);
            if (q0 < 0 || q0 + q.R > q.NS) { ok = false; continue; }
            for (int m = 0; m < 128; ++m) {
              const int f = t * 128 + m;
              if (f >= q.Ho * q.Wo) continue;
              for (int kk = 0; kk < 64; ++kk) {
                const int g = kc * 128 + a * 64 + kk;
                if (g >= q.Hi * q.Wi) continue;  // past the plane: the tensor copy fills zeros
                y[f] += (long)cache[(size_t)(q0 * q.Wo + m) * 64 + kk] * x[g];
              }
            }
          }
        }
      }
      for (int t = t0; t < t1; ++t) {
        int first, end;
        k_range(q.dmin, q.dmax, q.KB, t, first, end);
        if (seen[t] != end - first || end <= first) ok = false;
      }
    }
    for (size_t i = 0; i < y.size(); ++i)
      if (y[i] != ref[i]) { ok = false; break; }
  }
  if (!ok) {
    ++fails;
    printf("FAIL H=%lld W=%lld k=%dx%d p=%d,%d flip=%d NS=%d dmin=%d dmax=%d\n", (long long)c.H, (long long)c.W, kh,
           kw, c.ph, c.pw, (int)flip, q.NS, q.dmin, q.dmax);
  }
}

int main() {
  srand(1);
  for (int W : {8, 16, 32, 64})
    for (int H : {1, 3, 8, 9, 16, 31, 32, 33, 48, 64, 65, 100})
      for (int kh : {1, 3, 9, 13, 17, 21, 27, 31})
        for (int kw : {1, 3, 9, 15, 31})
          for (int phs : {0, 1, 2}) {
            const int pw = (kw - 1) / 2;
            const int ph = phs == 0 ? kh / 2 : phs == 1 ? 0 : kh - 1;
            for (bool flip : {false, true}) check(mk(4, 3, H, W, kh, kw, ph, pw), flip);
          }
  // the large-kernel inference layers
  for (int W : {16, 32, 64})
    for (int k : {13, 21, 27, 31}) {
      Conv c = mk(64, 384, W, W, k, k, k / 2, k / 2);
      for (bool flip : {false, true}) check(c, flip);
      Geo q;
      if (!make_geo(c, false, &q)) continue;
      KCfg kc{};
      size_t smem = 0;
      const bool has = plan_kernel(q, 64, &kc, &smem);
      printf("W=%d k=%d: NS=%d dmin=%d dmax=%d cached=%d cache=%zu B G=%d NG=%d nsets=%d ncols=%d stages=%d "
             "smem=%zu KB\n", W, k, q.NS, q.dmin, q.dmax, (int)has, cache_bytes(c, false), kc.G, kc.NG, kc.nsets,
             kc.ncols, kc.stages, smem / 1024);
    }
  printf("cases %d fails %d\n", cases, fails);
  return fails != 0 || cases == 0;
}
