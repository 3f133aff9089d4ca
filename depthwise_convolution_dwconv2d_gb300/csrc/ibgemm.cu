// Large-kernel depthwise forward / stride-1 grad-input on the 5th-generation
// tensor cores (tcgen05): fp16 / bf16 operands, fp32 accumulation in tensor
// memory.
//
// The MegEngine large-kernel depthwise article (section on the
// implicit-batched-GEMM algorithm) turns each channel of a large-kernel
// depthwise convolution into a GEMM by expanding the *filter* rather than
// the input: for channel c, with flattened output positions f = oh*Wo + ow
// and input positions g = ih*Wi + iw,
//   Y_c[f, n] = sum_g T_c[f, g] * X_c[g, n],
//   T_c[f, g] = w_c[ih - oh + ph][iw - ow + pw]   (0 outside the filter)
// so M = output positions, N = batch, K = input positions. The flop count
// exceeds the direct method's by roughly (plane area)/(filter area), which
// is why it pays only for large filters on small planes.
//
// Kernel structure (one CTA per SM, persistent over (channel, tile) units):
//  * warp 4 (one lane) streams X_c with TMA: per K step, 64 consecutive
//    input positions x nb samples, 128-byte swizzle, zero fill past the
//    plane and past the batch;
//  * warps 0-3 build the matching 128 x 64 block of T_c in shared memory in
//    the same swizzled K-major layout. Each 16-byte piece of a row is a run
//    of 8 consecutive taps of one filter row; eight copies of the padded
//    filter, shifted by 0..7 elements, make every such run an aligned
//    16-byte load;
//  * thread 0 issues the four K=16 tcgen05.mma of the step and commits them
//    to the stage's "free" barrier; after the tile's last step the builders
//    read the accumulator with tcgen05.ld, add the bias and store the tile.
// Only the K steps whose input rows reach the tile's outputs are visited.
//
// Every wait is bounded. A wait that gives up adds one to the library's
// timeout counter; the CTA then stops issuing work, waits (bounded) for its
// outstanding copies and MMAs, frees its tensor memory and returns.
#include <type_traits>

#include "plan.h"
#include "tile.cuh"
#include "tma.cuh"

namespace dwconv {
namespace ibg {
namespace {

constexpr int kBuilders = 128;  // warps 0-3: TMEM lanes 0..127 = rows of the M tile
constexpr int kThreads = kBuilders + 32;
constexpr int kM = 128, kKs = 64;  // M tile, K step (16-bit elements = 128 bytes)
constexpr int kABytes = kM * kKs * 2;
constexpr int kMaxStages = 4;

struct ICfg {
  int Hi, Wi, Ho, Wo;  // input / output planes
  int kh, kw, ph, pw;  // filter taps and padding of the correlation run
  int flip;            // grad-input: rotate the stored filter by 180 degrees
  int T;               // M tiles per channel
  int L;               // elements per padded, shifted filter row (L / 8 odd)
  int nb;              // MMA N (samples, multiple of 16, <= 256)
  int ncols;           // tensor-memory columns allocated (power of two >= 32)
  int S;               // pipeline stages
  uint32_t idesc;      // tcgen05 instruction descriptor
  uint32_t bbytes;     // bytes of one B stage (nb x 128)
  int64_t N, C;
  int64_t in_off;             // channel offset of the input slice
  int64_t out_ctot, out_off;  // channel count / offset of the output tensor
  int64_t units;              // C * T
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)1 << 16;            // leading byte offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset
  d |= (uint64_t)1 << 46;            // descriptor version
  d |= (uint64_t)2 << 61;            // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on bar once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(
                   tma::smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Barrier over the builder warps that also ORs a predicate across them.
__device__ __forceinline__ bool builders_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kBuilders)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void builders_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kBuilders) : "memory");
}

// Bounded wait; stops early when *abort is set (if abort is given). Counts a
// give-up in *timeouts (if given).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned int* timeouts,
                                         volatile int* abort) {
  for (uint32_t i = 0; i < tma::kWaitLimit; ++i) {
    if (tma::mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
  }
  if (timeouts) atomicAdd(timeouts, 1u);
  return false;
}

// K steps of tile t: 64-position blocks of the input plane whose rows reach
// the tile's outputs.
__host__ __device__ __forceinline__ void k_range(const ICfg& g, int t, int& kc_lo, int& kc_hi) {
  const int f0 = t * kM;
  int f1 = f0 + kM;
  if (f1 > g.Ho * g.Wo) f1 = g.Ho * g.Wo;
  const int oh_lo = f0 / g.Wo, oh_hi = (f1 - 1) / g.Wo;
  int ih_lo = oh_lo - g.ph, ih_hi = oh_hi - g.ph + g.kh - 1;
  if (ih_lo < 0) ih_lo = 0;
  if (ih_hi > g.Hi - 1) ih_hi = g.Hi - 1;
  kc_lo = ih_lo * g.Wi / kKs;
  kc_hi = ((ih_hi + 1) * g.Wi + kKs - 1) / kKs;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 1)
ibgemm_kernel(ICfg g, const __grid_constant__ CUtensorMap xmap, unsigned int* timeouts, const T* __restrict__ w,
              const T* __restrict__ bias, T* __restrict__ y, int accumulate_out) {
  extern __shared__ __align__(1024) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t full[kMaxStages], freeb[kMaxStages], dbar;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  // 1024-byte aligned: [A stages][B stages][shifted filter copies]
  unsigned char* base = smdyn + ((1024 - (tma::smem_u32(smdyn) & 1023)) & 1023);
  unsigned char* A = base;
  unsigned char* B = A + g.S * kABytes;
  T* SC = reinterpret_cast<T*>(B + g.S * g.bbytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < g.S; ++s) {
      tma::mbar_init(&full[s], 1);
      tma::mbar_init(&freeb[s], 1);
    }
    tma::mbar_init(&dbar, 1);
    tma::fence_init();
    abort_s = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     tma::smem_u32(&tmem_base_s)), "r"(g.ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  volatile int* abortp = &abort_s;
  const int64_t u0 = (int64_t)blockIdx.x * g.units / gridDim.x;
  const int64_t u1 = (int64_t)(blockIdx.x + 1) * g.units / gridDim.x;

  if (warp == 4) {
    // ---- producer: X_c blocks through the stage ring ----------------------
    if (lane == 0) {
      uint32_t step = 0;
      bool ok = true;
      for (int64_t u = u0; u < u1 && ok; ++u) {
        const int64_t c = u / g.T;
        const int t = (int)(u - c * g.T);
        int kc_lo, kc_hi;
        k_range(g, t, kc_lo, kc_hi);
        for (int kc = kc_lo; kc < kc_hi; ++kc) {
          const int s = step % g.S;
          const uint32_t use = step / g.S;
          if (use > 0 && !wait_bar(&freeb[s], (use - 1) & 1, timeouts, abortp)) { ok = false; break; }
          if (*abortp) { ok = false; break; }
          tma::mbar_expect_tx(&full[s], g.bbytes);
          tma::load_3d(B + s * g.bbytes, &xmap, kc * kKs, (int)(g.in_off + c), 0, &full[s]);
          ++step;
        }
      }
      if (!ok) *abortp = 1;
      // every issued copy must land before the CTA leaves
      const uint32_t first = step > (uint32_t)g.S ? step - g.S : 0;
      for (uint32_t k = first; k < step; ++k) wait_bar(&full[k % g.S], (k / g.S) & 1, nullptr, nullptr);
    }
    __syncwarp();
  } else {
    // ---- builders / MMA issuer / epilogue -------------------------------
    const int m = tid;
    uint32_t step = 0, tiles = 0;
    int64_t cur_c = -1;
    float bv = 0.f;
    bool fail = false, stop = false;
    for (int64_t u = u0; u < u1 && !stop; ++u) {
      const int64_t c = u / g.T;
      const int t = (int)(u - c * g.T);
      if (c != cur_c) {
        // eight copies of the padded filter rows, copy s shifted left by s:
        // SC[s][dy][i] = fr(dy, i + s), fr(dy, j) = w'[dy][j - (Wo - 1 - pw)]
        builders_sync();
        const T* wc = w + c * g.kh * g.kw;
        const int per = g.kh * g.L;
        for (int e = tid; e < 8 * per; e += kBuilders) {
          const int s = e / per, rem = e - s * per;
          const int dy = rem / g.L, i = rem - dy * g.L;
          const int b = i + s - (g.Wo - 1 - g.pw);
          float v = 0.f;
          if (b >= 0 && b < g.kw)
            v = g.flip ? ld(wc + (g.kh - 1 - dy) * g.kw + (g.kw - 1 - b)) : ld(wc + dy * g.kw + b);
          SC[e] = from_f<T>(v);
        }
        builders_sync();
        cur_c = c;
        bv = bias ? ld(bias + c) : 0.f;
      }
      int kc_lo, kc_hi;
      k_range(g, t, kc_lo, kc_hi);
      // this thread's row of the tile: output position f
      const int f = t * kM + m;
      const bool mvalid = f < g.Ho * g.Wo;
      const int oh = mvalid ? f / g.Wo : 0, ow = mvalid ? f - oh * g.Wo : 0;
      const int j0 = g.Wo - 1 - ow;
      const T* rowsrc = SC + (size_t)(j0 & 7) * g.kh * g.L + (j0 & ~7);
      unsigned char* arow_off = A + m * 128;
      for (int kc = kc_lo; kc < kc_hi; ++kc, ++step) {
        const int s = step % g.S;
        const uint32_t use = step / g.S;
        if (use > 0 && !wait_bar(&freeb[s], (use - 1) & 1, timeouts, abortp)) fail = true;
        unsigned char* arow = arow_off + s * kABytes;
        // 8 pieces of 8 input positions: kc*64 + 8j
        const int gpos = kc * kKs;
        int ih = gpos / g.Wi, iw = gpos - ih * g.Wi;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int dy = ih - oh + g.ph;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (mvalid && ih < g.Hi && dy >= 0 && dy < g.kh)
            v = *reinterpret_cast<const uint4*>(rowsrc + dy * g.L + iw);
          *reinterpret_cast<uint4*>(arow + ((j ^ (m & 7)) << 4)) = v;
          iw += 8;
          if (iw == g.Wi) { iw = 0; ++ih; }
        }
        tma::fence_async_smem();
        if (builders_sync_or(fail || *abortp)) { stop = true; break; }
        if (tid == 0) {
          if (!wait_bar(&full[s], use & 1, timeouts, abortp)) {
            fail = true;
            *abortp = 1;
          } else {
            tc_fence_after();
            const uint32_t a0 = tma::smem_u32(A + s * kABytes), b0 = tma::smem_u32(B + s * g.bbytes);
#pragma unroll
            for (int k = 0; k < kKs / 16; ++k)
              mma_f16(tmem, smem_desc(a0 + 32 * k), smem_desc(b0 + 32 * k), g.idesc,
                      (kc > kc_lo || k > 0) ? 1u : 0u);
            mma_commit(&freeb[s]);
          }
        }
      }
      if (stop) break;
      // epilogue: the accumulator is complete when the tile's MMAs are
      if (tid == 0) mma_commit(&dbar);
      bool okd = wait_bar(&dbar, tiles & 1, timeouts, abortp);
      ++tiles;
      okd = __all_sync(0xffffffffu, okd);
      if (!okd) {
        fail = true;
      } else {
        tc_fence_after();
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        T* yo = y + (g.out_off + c) * (int64_t)g.Ho * g.Wo + f;
        const int64_t nstride = g.out_ctot * (int64_t)g.Ho * g.Wo;
        for (int n0 = 0; n0 < g.nb; n0 += 16) {
          float v[16];
          tmem_ld16(trow + n0, v);
          if (mvalid) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int64_t n = n0 + i;
              if (n < g.N) {
                T* o = yo + n * nstride;
                const float val = v[i] + bv;
                *o = from_f<T>(accumulate_out ? val + ld_rw(o) : val);
              }
            }
          }
        }
      }
      tc_fence_before();
    }
    if (stop || fail) *abortp = 1;
    builders_sync();
    // all MMAs issued by thread 0 must be done before the memory is freed
    if (tid == 0 && step > 0) {
      mma_commit(&dbar);
      wait_bar(&dbar, tiles & 1, nullptr, nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(g.ncols) : "memory");
}

// Padded filter row length: at least Wo + Wi - 1 + 8, a multiple of 8 with
// L / 8 odd (the eight shifted copies then start in different bank groups).
int row_len(int Wi, int Wo) {
  int L = tile::round_up(Wo + Wi - 1 + 8, 8);
  if ((L / 8) % 2 == 0) L += 8;
  return L;
}

size_t smem_bytes(int S, int nb, int kh, int L) {
  return 1024 + (size_t)S * (kABytes + (size_t)nb * 128) + (size_t)8 * kh * L * 2;
}

// Geometry of the correlation the kernel runs: the forward as given, the
// grad-input as a correlation of grad_out with the rotated filter and
// padding k - 1 - p.
struct Geo {
  int Hi, Wi, Ho, Wo, ph, pw;
};

Geo geo_of(const Conv& c, bool flip) {
  if (!flip) return Geo{(int)c.H, (int)c.W, (int)c.Ho, (int)c.Wo, c.ph, c.pw};
  return Geo{(int)c.Ho, (int)c.Wo, (int)c.H, (int)c.W, c.kh - 1 - c.ph, c.kw - 1 - c.pw};
}

int stages_for(const Conv& c, const Geo& q) {
  const int nb = tile::round_up(c.N, 16);
  const int L = row_len(q.Wi, q.Wo);
  for (int S = kMaxStages; S >= 2; --S)
    if (smem_bytes(S, nb, c.kh, L) <= 227 * 1024) return S;
  return 0;
}

template <typename T>
cudaError_t run(const Conv& c, bool flip, const void* in, const void* w, const void* bias, void* out, bool acc,
                cudaStream_t s) {
  const Geo q = geo_of(c, flip);
  if (reinterpret_cast<uintptr_t>(in) % 16 != 0) return cudaErrorNotSupported;
  ICfg g{};
  g.Hi = q.Hi; g.Wi = q.Wi; g.Ho = q.Ho; g.Wo = q.Wo;
  g.kh = c.kh; g.kw = c.kw; g.ph = q.ph; g.pw = q.pw;
  g.flip = flip;
  g.T = (g.Ho * g.Wo + kM - 1) / kM;
  g.L = row_len(g.Wi, g.Wo);
  g.nb = tile::round_up(c.N, 16);
  g.ncols = 32;
  while (g.ncols < g.nb) g.ncols *= 2;
  g.S = stages_for(c, q);
  if (g.S == 0) return cudaErrorInvalidConfiguration;
  const bool bf = std::is_same<T, __nv_bfloat16>::value;
  // D fp32 (bits 4-5 = 1); A, B fp16 (0) or bf16 (1) in bits 7-9 / 10-12;
  // both K-major (bits 15, 16 = 0); N >> 3 in bits 17-22; M >> 4 in bits 24-28
  g.idesc = (1u << 4) | ((bf ? 1u : 0u) << 7) | ((bf ? 1u : 0u) << 10) | ((uint32_t)(g.nb >> 3) << 17) |
            ((uint32_t)(kM >> 4) << 24);
  g.bbytes = (uint32_t)g.nb * 128;
  g.N = c.N;
  g.C = c.C;
  int64_t in_ctot;
  if (flip) {  // input: the grad_out slice; output: grad_in
    in_ctot = c.ctot; g.in_off = c.off; g.out_ctot = c.C; g.out_off = 0;
  } else {
    in_ctot = c.C; g.in_off = 0; g.out_ctot = c.ctot; g.out_off = c.off;
  }
  g.units = c.C * g.T;
  // input as [N][channels][Hi*Wi]: box = 64 positions x 1 channel x nb samples
  alignas(64) CUtensorMap map{};
  if (!tma::encode_3d_sw128(&map, in, c.dtype, (uint64_t)g.Hi * g.Wi, (uint64_t)in_ctot, (uint64_t)c.N,
                            (uint32_t)kKs, 1, (uint32_t)g.nb))
    return cudaErrorInvalidValue;
  const size_t smem = smem_bytes(g.S, g.nb, g.kh, g.L);
  auto kern = ibgemm_kernel<T>;
  cudaError_t e = tile::set_smem(kern, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, occ = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem)) != cudaSuccess) return e;
  // resident CTAs must never need more than the 512 tensor-memory columns
  if (occ < 1 || occ * g.ncols > 512) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)sms * occ;
  if (grid > g.units) grid = g.units;
  if (grid < 1) return cudaSuccess;
  kern<<<(int)grid, kThreads, smem, s>>>(g, map, tma::timeout_counter(), (const T*)w, (const T*)bias, (T*)out,
                                         acc ? 1 : 0);
  return cudaGetLastError();
}

bool geo_supported(const Conv& c, bool flip) {
  if (c.dtype != DWCONV_F16 && c.dtype != DWCONV_BF16) return false;  // tensor cores for 16-bit data only
  if (c.sh != 1 || c.sw != 1 || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if (c.kh < 9 || c.kw < 9) return false;  // smaller filters stay on the direct kernels
  if (c.ph > c.kh - 1 || c.pw > c.kw - 1 || c.Ho < 1 || c.Wo < 1) return false;
  if (c.N < 1 || c.N > 256) return false;
  const Geo q = geo_of(c, flip);
  // input rows of 16-byte multiples (8-element pieces never straddle rows)
  if (q.Wi % 8 != 0 || q.Wi > 128 || q.Wo > 128 || q.Hi > 128 || q.Ho > 128) return false;
  return stages_for(c, q) > 0;
}

}  // namespace

bool fwd_supported(const Conv& c) { return geo_supported(c, false); }
bool bwd_data_supported(const Conv& c) { return geo_supported(c, true); }

cudaError_t fwd(const Conv& c, const void* x, const void* w, const void* b, void* y, cudaStream_t s) {
  if (c.dtype == DWCONV_F16) return run<__half>(c, false, x, w, b, y, false, s);
  if (c.dtype == DWCONV_BF16) return run<__nv_bfloat16>(c, false, x, w, b, y, false, s);
  return cudaErrorInvalidValue;
}

cudaError_t bwd_data(const Conv& c, const void* gy, const void* w, void* gx, bool acc, cudaStream_t s) {
  if (c.dtype == DWCONV_F16) return run<__half>(c, true, gy, w, nullptr, gx, acc, s);
  if (c.dtype == DWCONV_BF16) return run<__nv_bfloat16>(c, true, gy, w, nullptr, gx, acc, s);
  return cudaErrorInvalidValue;
}

}  // namespace ibg
}  // namespace dwconv
