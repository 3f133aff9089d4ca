// Large-kernel weight gradient for fp16 / bf16 data on the 5th-generation
// tensor cores (tcgen05, fp32 accumulation in tensor memory).
//
// The MegEngine large-kernel depthwise article (section on the implicit
// batched GEMM) runs large depthwise filters on the tensor cores by turning
// each channel into a GEMM whose Toeplitz operand is expanded on chip. The
// weight gradient of one channel has the same structure:
//   gw[a][b] = sum_{n, oh} sum_iw  X[a][(n, oh, iw)] * G[(n, oh, iw)][b]
//   X[a][(n, oh, iw)] = x~[n][oh + a][iw]          (rows of the padded x plane)
//   G[(n, oh, iw)][b] = gy[n][oh][iw - b + shift]  (a Toeplitz of grad_out rows)
// so M = filter rows (padded to 64), N = filter columns (32, in reverse
// order), K = samples x output rows x input columns.
//
// Neither operand is copied into a GEMM layout:
//  * The x plane of a sample is loaded by one TMA copy into shared memory as
//    8-column blocks, each block holding every row at a 16-byte stride (the
//    no-swizzle K-major core-matrix layout). The A operand for output row oh
//    is then the same buffer seen from row oh: a descriptor start address
//    16 * oh bytes further on.
//  * Reversing the filter columns (n' = 31 - b) makes the 8 x 8 core matrix
//    (n'-group g, K-block j) of the Toeplitz depend on j + g only. So a
//    grad_out row is stored once as eight copies shifted by 0..7 elements,
//    interleaved 16 bytes at a time: block t of that storage is exactly core
//    matrix j + g = t, and the B operand is a descriptor with both strides
//    equal to 128 bytes. Builder warps write these copies from the staged
//    grad_out plane, a group of eight output rows at a time.
// For every output row, (columns / 16) MMAs of 64 x 32 x 16 accumulate into
// one tensor-memory tile; after the last sample of a (channel, batch chunk)
// unit, two warps read the tile (D row a sits in lane 32 * (a / 16) +
// a % 16) and write one partial per (chunk, channel) -- the same partials as
// the other weight-gradient kernels, summed in index order by the second
// pass.
//
// Warp roles, connected by mbarriers only: warp 0 issues the MMAs (one
// elected lane), warp 1 issues the TMA copies (one lane), warps 2-7 build the
// shifted copies (warp 2 also sums grad_out for the bias gradient), and
// warps 4-5 read the accumulator at the end of a unit. Every wait is
// bounded; a wait that gives up counts in the library's timeout counter and
// raises the CTA's abort flag, every role leaves its loop, the issuer and
// the producer wait (bounded) for their operations in flight, and the CTA
// frees its tensor memory and returns.
#include "plan.h"
#include "tile.cuh"
#include "tma.cuh"

namespace dwconv {
namespace wtc {
namespace {

constexpr int kThreads = 256;
constexpr int kM = 64, kN = 32;  // MMA shape: filter rows (padded), filter columns (reversed)
constexpr int kGroup = 8;        // output rows per shifted-copy buffer
constexpr int kBuildWarps = 6;   // warps 2..7
constexpr int kBuilders = kBuildWarps * 32;
constexpr unsigned kSleepNs = 64;

struct WCfg {
  int K, pad, P8;
  int H, W, Ho, Wo;
  int nk;             // 16-column K steps per output row
  int RT;             // rows of the x tile (Ho + 63: the A operand of the last row reads 64 rows)
  int nblkB;          // 128-byte blocks per shifted-copy row (2 nk + 3)
  int delta;          // grad_out column of shifted-copy block 0, copy 0, element 0
  int ngroups;        // groups of kGroup output rows
  uint32_t xbytes;    // one x tile (16 * RT * 2 nk)
  uint32_t gbytes;    // one staged grad_out plane (Ho * Wo * 2)
  uint32_t sbytes;    // one shifted-copy buffer (kGroup * nblkB * 128)
  uint32_t xoff, goff, soff;           // shared-memory offsets of buffer 0 of each kind
  uint32_t xstr, gstr, sstr;           // distance to buffer 1 (runtime-indexed arrays would
                                       // move the launch parameters to local memory)
  uint32_t idesc;
  int chunks, nb;
  int64_t units;      // C * chunks
  int64_t gy_ctot, gy_off;
};

__device__ __forceinline__ uint32_t su32(const void* p) { return tma::smem_u32(p); }

// Shared-memory matrix descriptor, no swizzle, K-major: leading byte offset =
// stride between core matrices along K, stride byte offset = stride between
// 8-row groups.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  return d;
}

__device__ __forceinline__ void mma_ss(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(su32(bar))
               : "memory");
}

__device__ __forceinline__ void arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(su32(bar)) : "memory");
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// Bounded wait that gives up early once the CTA aborts.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, unsigned int* timeouts,
                                         volatile int* abort, unsigned sleep_ns = 0) {
  for (uint32_t i = 0; i < tma::kWaitLimit; ++i) {
    if (tma::mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if (sleep_ns) __nanosleep(sleep_ns);
  }
  if (timeouts) atomicAdd(timeouts, 1u);
  return false;
}

// Walk of a CTA's steps: units u = blockIdx.x, blockIdx.x + gridDim.x, ...;
// unit u is channel u % C, batch chunk u / C; a step is one sample of it.
struct Steps {
  int64_t u, units, C, N, stride;
  int nb, s, ns;
  __device__ __forceinline__ Steps(int64_t u0, int64_t stride_, int64_t units_, int64_t C_, int64_t N_, int nb_)
      : u(u0), units(units_), C(C_), N(N_), stride(stride_), nb(nb_), s(0) {
    ns = count();
    while (u < units && ns == 0) {  // (none when chunks = ceil(N / nb))
      u += stride;
      ns = count();
    }
  }
  __device__ __forceinline__ int count() const {
    if (u >= units) return 0;
    const int64_t n0 = (u / C) * nb;
    const int64_t left = N - n0;
    return (int)(left < nb ? (left > 0 ? left : 0) : nb);
  }
  __device__ __forceinline__ bool more() const { return u < units; }
  __device__ __forceinline__ int64_t ch() const { return u % C; }
  __device__ __forceinline__ int64_t chunk() const { return u / C; }
  __device__ __forceinline__ int64_t n() const { return chunk() * nb + s; }
  __device__ __forceinline__ bool last() const { return s + 1 >= ns; }
  // next step; units without samples are skipped
  __device__ __forceinline__ void next() {
    if (++s >= ns) {
      s = 0;
      do {
        u += stride;
        ns = count();
      } while (u < units && ns == 0);
    }
  }
};

template <bool BF>
__global__ void __launch_bounds__(kThreads, 1)
wgrad_tc_kernel(Conv c, WCfg g, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap gmap,
                unsigned int* timeouts, float* __restrict__ ws) {
  extern __shared__ __align__(1024) unsigned char smdyn[];
  __shared__ __align__(8) uint64_t xfull[2], xfree[2], sfull[2], sfree[2], dfull, dfree, done;
  __shared__ uint32_t tmem_s;
  __shared__ int abort_s;
  unsigned char* base = smdyn + ((1024 - (su32(smdyn) & 1023)) & 1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      tma::mbar_init(&xfull[i], 1);
      tma::mbar_init(&xfree[i], 1 + kBuildWarps);
      tma::mbar_init(&sfull[i], kBuildWarps);
      tma::mbar_init(&sfree[i], 1);
    }
    tma::mbar_init(&dfull, 1);
    tma::mbar_init(&dfree, 2);
    tma::mbar_init(&done, 1);
    tma::fence_init();
    abort_s = 0;
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 32;\n" ::"r"(su32(&tmem_s))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  const uint32_t tmem = tmem_s;
  volatile int* abortp = &abort_s;
  const int K = g.K, KK = K * K;

  if (warp == 1) {
    // ---- producer: x tile and grad_out plane of each step -----------------
    if (lane == 0) {
      uint32_t k = 0;
      for (Steps st(blockIdx.x, gridDim.x, g.units, c.C, c.N, g.nb); st.more() && !*abortp; st.next(), ++k) {
        const int slot = k & 1;
        if (k >= 2 && !wait_bar(&xfree[slot], ((k >> 1) - 1) & 1, timeouts, abortp, kSleepNs)) {
          *abortp = 1;
          break;
        }
        const int64_t n = st.n(), ch = st.ch();
        tma::mbar_expect_tx(&xfull[slot], g.xbytes + g.gbytes);
        tma::load_4d(base + g.xoff + slot * g.xstr, &xmap, 0, -g.pad, -(g.P8 / 8), (int)(n * c.C + ch), &xfull[slot]);
        tma::load_3d(base + g.goff + slot * g.gstr, &gmap, 0, 0, (int)(n * g.gy_ctot + g.gy_off + ch),
                     &xfull[slot]);
      }
      // every issued copy lands before the CTA leaves
      const uint32_t first = k > 2 ? k - 2 : 0;
      for (uint32_t j = first; j < k; ++j) wait_bar(&xfull[j & 1], (j >> 1) & 1, nullptr, nullptr);
    }
    __syncwarp();
  } else if (warp == 0) {
    // ---- MMA issuer -----------------------------------------------------------
    const uint32_t lboA = (uint32_t)g.RT * 16;
    uint32_t k = 0, grp = 0, unit_no = 0;
    bool ok = true;
    Steps st(blockIdx.x, gridDim.x, g.units, c.C, c.N, g.nb);
    while (st.more() && ok) {
      // the accumulator is free once the previous unit's epilogue read it
      if (unit_no > 0) ok = wait_bar(&dfree, (unit_no - 1) & 1, timeouts, abortp);
      bool first_mma = true;
      bool unit_end = false;
      while (ok && !unit_end) {
        const int slot = k & 1;
        ok = wait_bar(&xfull[slot], (k >> 1) & 1, timeouts, abortp);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        const uint32_t xa = su32(base + g.xoff + slot * g.xstr);
        for (int gi = 0; gi < g.ngroups && ok; ++gi, ++grp) {
          const int sslot = grp & 1;
          ok = wait_bar(&sfull[sslot], (grp >> 1) & 1, timeouts, abortp);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
          const uint32_t sa = su32(base + g.soff + sslot * g.sstr);
          const int oh0 = gi * kGroup;
          const int oh1 = (oh0 + kGroup) < g.Ho ? (oh0 + kGroup) : g.Ho;
          // the unit's first MMA overwrites the accumulator, the rest add.
          // The whole warp walks the loop (descriptors stay warp-uniform) and
          // one elected lane issues each MMA.
          uint32_t acc = first_mma ? 0u : 1u;
          const bool leader = elect_one();
          const uint64_t astep = (uint64_t)((2u * lboA) >> 4), bstep = 256u >> 4;
          for (int oh = oh0; oh < oh1; ++oh) {
            uint64_t ad = sdesc(xa + 16u * oh, lboA, 128);
            uint64_t bd = sdesc(sa + (uint32_t)(oh - oh0) * g.nblkB * 128u, 128, 128);
#pragma unroll 4
            for (int jj = 0; jj < g.nk; ++jj) {
              if (leader) mma_ss(tmem, ad, bd, g.idesc, acc);
              acc = 1u;
              ad += astep;
              bd += bstep;
            }
          }
          if (leader) commit(&sfree[sslot]);
          __syncwarp();
          first_mma = false;
        }
        if (!ok) break;
        if (elect_one()) commit(&xfree[slot]);
        __syncwarp();
        unit_end = st.last();
        st.next();
        ++k;
      }
      if (!ok) break;
      if (elect_one()) commit(&dfull);
      __syncwarp();
      ++unit_no;
    }
    if (!ok) *abortp = 1;
    // every MMA is done before the tensor memory is freed
    if (elect_one()) commit(&done);
    __syncwarp();
    wait_bar(&done, 0, nullptr, nullptr);
    __syncwarp();
  } else {
    // ---- builders (warps 2..7), epilogue (warps 4, 5) --------------------------
    const int bt = tid - 64;  // 0..191
    uint32_t k = 0, grp = 0, unit_no = 0;
    float bsum = 0.f;
    bool ok = true;
    for (Steps st(blockIdx.x, gridDim.x, g.units, c.C, c.N, g.nb); st.more() && ok; st.next(), ++k) {
      const int slot = k & 1;
      ok = wait_bar(&xfull[slot], (k >> 1) & 1, timeouts, abortp, kSleepNs);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      const unsigned short* gp = reinterpret_cast<const unsigned short*>(base + g.goff + slot * g.gstr);
      if (warp == 2) {
        // bias gradient: one warp sums every grad_out value, in a fixed order
        for (int e = lane; e < g.Ho * g.Wo; e += 32)
          bsum += BF ? __bfloat162float(__ushort_as_bfloat16(gp[e])) : __half2float(__ushort_as_half(gp[e]));
      }
      const int wch = g.Wo / 8;  // 16-byte chunks per grad_out row
      for (int gi = 0; gi < g.ngroups && ok; ++gi, ++grp) {
        const int sslot = grp & 1;
        if (grp >= 2) {
          ok = wait_bar(&sfree[sslot], ((grp >> 1) - 1) & 1, timeouts, abortp, kSleepNs);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        }
        const int oh0 = gi * kGroup;
        const int nrows = (g.Ho - oh0) < kGroup ? (g.Ho - oh0) : kGroup;
        uint4* sp = reinterpret_cast<uint4*>(base + g.soff + sslot * g.sstr);
        // unit e = (row r, block blk, copy s): grad_out[oh0 + r][o .. o + 7],
        // o = 8 blk + s + delta, from the two 16-byte chunks around it (zero
        // chunks outside the row). Consecutive threads write consecutive units.
        const int runits = g.nblkB * 8;
        for (int e = bt; e < nrows * runits; e += kBuilders) {
          const int r = e / runits;
          const int o = (e - r * runits) + g.delta;  // 8 blk + s + delta
          const int q = ((o + 64) >> 3) - 8;         // floor(o / 8) (o > -64)
          const int rr = o & 7;
          const uint4* row = reinterpret_cast<const uint4*>(gp + (oh0 + r) * g.Wo);
          const uint4 z = make_uint4(0, 0, 0, 0);
          const uint4 c0 = ((unsigned)q < (unsigned)wch) ? row[q] : z;
          const uint4 c1 = ((unsigned)(q + 1) < (unsigned)wch) ? row[q + 1] : z;
          const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
          // words k .. k + 4 (k = rr / 2), then a 16-bit shift for odd rr
          const int k = rr >> 1;
          uint32_t v[5];
#pragma unroll
          for (int i = 0; i < 5; ++i) {
            const uint32_t lo = (k & 1) ? w[(i + 1) & 7] : w[i];
            const uint32_t hi = (k & 1) ? w[(i + 3) & 7] : w[(i + 2) & 7];
            v[i] = (k & 2) ? hi : lo;
          }
          const uint32_t sh = (rr & 1) ? 16u : 0u;
          sp[e] = make_uint4(__funnelshift_r(v[0], v[1], sh), __funnelshift_r(v[1], v[2], sh),
                             __funnelshift_r(v[2], v[3], sh), __funnelshift_r(v[3], v[4], sh));
        }
        // generic-proxy writes, read next by the tensor core (async proxy)
        tma::fence_async_smem();
        __syncwarp();
        if (lane == 0) arrive(&sfull[sslot]);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) arrive(&xfree[slot]);
      if (st.last()) {
        // end of the unit: the accumulator (warps 4, 5) and the bias sum
        const int64_t ch = st.ch(), q = st.chunk();
        float* dstp = ws + (q * c.OC() + ch) * (KK + 1);
        if (warp == 4 || warp == 5) {
          ok = wait_bar(&dfull, unit_no & 1, timeouts, abortp);
          if (__all_sync(0xffffffffu, ok)) {
            asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
            uint32_t v[32];
            asm volatile(
                "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
                  "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
                  "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]),
                  "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]),
                  "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                : "r"(tmem + ((uint32_t)((warp - 4) * 32) << 16)));
            asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
            // lane l of warp 4 + h holds filter row a = 16 h + l (l < 16);
            // column n' holds filter column b = 31 - n'
            const int a = 16 * (warp - 4) + lane;
            if (lane < 16 && a < K) {
#pragma unroll
              for (int nn = 0; nn < 32; ++nn) {
                const int b = kN - 1 - nn;
                if (b < K) dstp[a * K + b] = __uint_as_float(v[nn]);
              }
            }
            asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
          } else {
            ok = false;
          }
          __syncwarp();
          if (lane == 0) arrive(&dfree);
        }
        if (warp == 2) {
          float bv = bsum;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) bv += __shfl_xor_sync(0xffffffffu, bv, o);
          bsum = 0.f;
          if (lane == 0) dstp[KK] = bv;
        }
        ++unit_no;
      }
    }
    if (!ok) *abortp = 1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 32;\n" ::"r"(tmem) : "memory");
}

bool plan(const Conv& c, WCfg* out, size_t* smem_out) {
  WCfg g{};
  g.K = c.kh;
  g.pad = c.ph;
  g.P8 = (c.ph + 7) / 8 * 8;
  g.H = (int)c.H; g.W = (int)c.W; g.Ho = (int)c.Ho; g.Wo = (int)c.Wo;
  // x tile columns: every input column a nonzero Toeplitz entry meets
  const int cols = g.Wo + g.K - 1 - g.pad + g.P8;
  g.nk = (cols + 15) / 16;
  g.RT = g.Ho + kM - 1;
  g.nblkB = 2 * g.nk + 3;
  g.delta = g.pad - g.P8 - (kN - 1);
  g.ngroups = (g.Ho + kGroup - 1) / kGroup;
  g.xbytes = 16u * (uint32_t)g.RT * (uint32_t)(2 * g.nk);
  g.gbytes = (uint32_t)(g.Ho * g.Wo * 2);
  g.sbytes = (uint32_t)(kGroup * g.nblkB * 128);
  auto al = [](uint32_t v) { return (v + 1023u) / 1024u * 1024u; };
  g.xstr = al(g.xbytes);
  g.gstr = al(g.gbytes);
  g.sstr = al(g.sbytes);
  g.xoff = 0;
  g.goff = 2 * g.xstr;
  g.soff = g.goff + 2 * g.gstr;
  const uint32_t off = g.soff + 2 * g.sstr;
  const size_t smem = (size_t)off + 1024;
  if (smem > 200 * 1024) return false;
  if (out) *out = g;
  if (smem_out) *smem_out = smem;
  return true;
}

}  // namespace

bool supported(const Conv& c) {
  if (c.dtype != DWCONV_F16 && c.dtype != DWCONV_BF16) return false;
  if (!c.planes32()) return false;
  if (c.kh != c.kw || c.kh < 7 || c.kh > kN || (c.kh & 1) == 0) return false;
  if (c.sh != 1 || c.sw != 1 || c.dh != 1 || c.dw != 1 || c.m != 1) return false;
  if (c.ph != c.pw || c.ph > c.kh - 1) return false;
  // 16-byte rows for the TMA copies of x and grad_out; box limits
  if (c.W % 8 != 0 || c.Wo % 8 != 0 || c.H > 128 || c.W > 128 || c.Ho > 128 || c.Wo > 128) return false;
  if (c.Ho + kM - 1 > 256) return false;
  return plan(c, nullptr, nullptr);
}

cudaError_t wgrad(const Conv& c, const void* x, const void* gy, float* ws, int chunks, cudaStream_t s) {
  if ((reinterpret_cast<uintptr_t>(x) % 16) != 0 || (reinterpret_cast<uintptr_t>(gy) % 16) != 0)
    return cudaErrorNotSupported;
  WCfg g;
  size_t smem = 0;
  if (!plan(c, &g, &smem)) return cudaErrorInvalidConfiguration;
  g.chunks = chunks;
  g.nb = (int)((c.N + chunks - 1) / chunks);
  g.units = c.C * chunks;
  g.gy_ctot = c.ctot;
  g.gy_off = c.off;
  const bool bf = c.dtype == DWCONV_BF16;
  // D fp32 (bit 4); A, B fp16 (0) or bf16 (1) in bits 7-9 / 10-12; both
  // K-major; N >> 3 in bits 17-22; M >> 4 in bits 24-28
  g.idesc = (1u << 4) | ((bf ? 1u : 0u) << 7) | ((bf ? 1u : 0u) << 10) | ((uint32_t)(kN >> 3) << 17) |
            ((uint32_t)(kM >> 4) << 24);
  // x as (8 elements, rows, 8-column blocks, planes): box (8, RT, 2 nk, 1)
  // lands as [block][row][8] -- the K-major core-matrix layout of A
  alignas(64) CUtensorMap xmap{}, gmap{};
  {
    const uint64_t dims[4] = {8, (uint64_t)c.H, (uint64_t)(c.W / 8), (uint64_t)(c.N * c.C)};
    const uint64_t strides[3] = {(uint64_t)c.W * 2, 16, (uint64_t)c.H * c.W * 2};
    const uint32_t box[4] = {8, (uint32_t)g.RT, (uint32_t)(2 * g.nk), 1};
    if (!tma::encode_strided(&xmap, x, c.dtype, 4, dims, strides, box)) return cudaErrorNotSupported;
  }
  {
    const uint64_t dims[3] = {(uint64_t)c.Wo, (uint64_t)c.Ho, (uint64_t)(c.N * c.ctot)};
    const uint64_t strides[2] = {(uint64_t)c.Wo * 2, (uint64_t)c.Ho * c.Wo * 2};
    const uint32_t box[3] = {(uint32_t)c.Wo, (uint32_t)c.Ho, 1};
    if (!tma::encode_strided(&gmap, gy, c.dtype, 3, dims, strides, box)) return cudaErrorNotSupported;
  }
  cudaError_t e;
  auto kern = bf ? wgrad_tc_kernel<true> : wgrad_tc_kernel<false>;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  int dev = 0, sms = 152;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // CTAs per SM from shared memory, registers and threads (tensor memory:
  // 32 columns each, never the limit)
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  int smem_sm = 0, regs_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess) return e;
  const int by_smem = smem_sm / (int)(smem + fa.sharedSizeBytes + 1024);
  const int by_regs = regs_sm / ((kThreads / 32) * ((fa.numRegs * 32 + 255) / 256 * 256));
  int per_sm = by_smem < by_regs ? by_smem : by_regs;
  if (per_sm > 4) per_sm = 4;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)sms * per_sm;
  if (grid > g.units) grid = g.units;
  if (grid < 1) return cudaSuccess;
  kern<<<(int)grid, kThreads, smem, s>>>(c, g, xmap, gmap, tma::timeout_counter(), ws);
  return cudaGetLastError();
}

}  // namespace wtc
}  // namespace dwconv
