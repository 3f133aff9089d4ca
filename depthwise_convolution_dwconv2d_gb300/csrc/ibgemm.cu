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
// Kernel structure (persistent CTAs over (channel, tile) units; warp roles
// hand work to one another through mbarriers only):
//  * producer (warp 12, one lane): per K step, TMA-loads 64 consecutive input
//    positions x nb samples of X_c into a shared-memory B stage, 128-byte
//    swizzle (the K-major operand layout), zero fill past the plane and the
//    batch;
//  * builders (warps 0-7): write the matching 128 x 64 block of T_c into a
//    tensor-memory A stage (tcgen05.st; lane = output position, two 16-bit
//    taps per column); warp w writes lanes 32*(w%4).. and half w/4 of the
//    taps. Each 8-tap piece of a row is a run of consecutive taps of one
//    filter row, one aligned 16-byte load from eight copies of the padded
//    filter shifted by 0..7 elements;
//  * MMA issuer (warp 13, one lane): four K=16 tcgen05.mma per step (A from
//    tensor memory, B from shared memory) into one of two fp32 accumulators,
//    then commits that free the stages and, after a tile's last step, hand
//    the accumulator to the epilogue;
//  * epilogue (warps 8-11): tcgen05.ld of the accumulator, bias, store.
// Only the K steps whose input rows reach the tile's outputs are visited.
//
// Every wait is bounded. A wait that gives up adds one to the library's
// timeout counter and raises the CTA's abort flag; from then on every role
// runs through its loops without waiting or issuing work (so the builders'
// named barriers stay matched), the issuer and the producer wait (bounded)
// for their outstanding MMAs and copies, the CTA frees its tensor memory and
// returns.
#include <type_traits>

#include "plan.h"
#include "tile.cuh"
#include "tma.cuh"

namespace dwconv {
namespace ibg {
namespace {

constexpr int kBuilders = 256;  // warps 0-7: rows of the M tile (TMEM lanes), two halves of K
constexpr int kEpiWarp0 = 8;    // warps 8-11: epilogue
constexpr int kProducerWarp = 12;
constexpr int kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int kM = 128;            // M tile (output positions)
constexpr int kAtom = 64;          // input positions per 128-byte swizzle atom (= 32 TMEM columns)
constexpr int kAtoms = 2;          // atoms per K step
constexpr int kKs = kAtom * kAtoms;  // K step (input positions)
constexpr int kS = 2;              // pipeline stages: A in tensor memory, B in shared memory
constexpr unsigned kSleepNs = 64;  // poll interval of the waits off the critical path

struct ICfg {
  int Hi, Wi, Ho, Wo;  // input / output planes
  int kh, kw, ph, pw;  // filter taps and padding of the correlation run
  int flip;            // grad-input: rotate the stored filter by 180 degrees
  int T;               // M tiles per channel
  int L;               // elements per padded, shifted filter row (L / 8 odd)
  int nb;              // MMA N (samples, multiple of 16, <= 256)
  int ncols;           // tensor-memory columns allocated (power of two >= 32)
  int acc_cols;        // columns per accumulator (nb rounded up to 32)
  int nacc;            // accumulators (2: the epilogue overlaps the next tile; 1 for nb > 128)
  int acol;            // first tensor-memory column of the A stages (after the accumulators)
  uint32_t idesc;      // tcgen05 instruction descriptor
  uint32_t bbytes;     // bytes of one B atom (nb x 128); a stage holds kAtoms of them
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

// D (tensor memory) (+)= A (tensor memory) x B (shared memory)^T
__device__ __forceinline__ void mma_f16_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(dtmem),
      "r"(atmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// One lane of the (converged) warp; the others get false.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// Named barrier over the builder warps.
__device__ __forceinline__ void builders_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kBuilders) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(tma::smem_u32(bar)) : "memory");
}

// Bounded wait; stops early when *abort is set (if abort is given). Counts a
// give-up in *timeouts (if given). Roles whose waits are hidden by the
// pipeline depth sleep between polls (sleep_ns > 0) so that they leave the
// issue slots and the barrier unit to the MMA issuer.
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

// Walk over this CTA's units u0..u1-1 as (channel c, tile t) without a
// division per unit.
struct Units {
  int64_t c, u, u1;
  int t, T;
  __device__ __forceinline__ Units(int64_t u0_, int64_t u1_, int T_) : u(u0_), u1(u1_), T(T_) {
    c = u0_ / T_;
    t = (int)(u0_ - c * T_);
  }
  __device__ __forceinline__ bool more() const { return u < u1; }
  __device__ __forceinline__ void next() {
    ++u;
    if (++t == T) { t = 0; ++c; }
  }
};

// Stage ring position: stage index and the parity of its current use.
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  bool wrapped = false;  // every stage has been used at least once
  __device__ __forceinline__ void next() {
    if (++s == kS) { s = 0; ph ^= 1; wrapped = true; }
  }
};

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
ibgemm_kernel(ICfg g, const __grid_constant__ CUtensorMap xmap, unsigned int* timeouts, const T* __restrict__ w_,
              const T* __restrict__ bias, T* __restrict__ y, int accumulate_out) {
  extern __shared__ __align__(1024) unsigned char smdyn[];
  // fullB[s]: the producer's expect_tx arrival and the copy's bytes; afull[s]:
  // the builders' 256 arrivals; freeS[s]: the MMAs that read stage s are done
  __shared__ __align__(8) uint64_t fullB[kS], afull[kS], freeS[kS], accfull[2], accfree[2], done;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  // 1024-byte aligned: [B stages][shifted filter copies]
  unsigned char* B = smdyn + ((1024 - (tma::smem_u32(smdyn) & 1023)) & 1023);
  const uint32_t sbytes = kAtoms * g.bbytes;  // bytes per B stage
  T* SC = reinterpret_cast<T*>(B + kS * sbytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kS; ++s) {
      tma::mbar_init(&fullB[s], 1);
      tma::mbar_init(&afull[s], kBuilders);
      tma::mbar_init(&freeS[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tma::mbar_init(&accfull[s], 1);
      tma::mbar_init(&accfree[s], 128);
    }
    tma::mbar_init(&done, 1);
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

  if (warp == kProducerWarp) {
    // ---- producer: X_c blocks through the B ring --------------------------
    if (lane == 0) {
      Ring r;
      uint32_t issued = 0;
      for (Units w(u0, u1, g.T); w.more(); w.next()) {
        const int64_t c = w.c;
        int kc_lo, kc_hi;
        k_range(g, w.t, kc_lo, kc_hi);
        for (int kc = kc_lo; kc < kc_hi && !*abortp; ++kc, r.next()) {
          if (r.wrapped && !wait_bar(&freeS[r.s], r.ph ^ 1, timeouts, abortp, kSleepNs)) { *abortp = 1; break; }
          tma::mbar_expect_tx(&fullB[r.s], sbytes);
#pragma unroll
          for (int a = 0; a < kAtoms; ++a)
            tma::load_3d(B + r.s * sbytes + a * g.bbytes, &xmap, kc * kKs + a * kAtom, (int)(g.in_off + c), 0,
                         &fullB[r.s]);
          ++issued;
        }
      }
      // every issued copy must land before the CTA leaves: the last kS uses
      // of the stages (fullB phases complete on the copy's bytes alone)
      const uint32_t first = issued > (uint32_t)kS ? issued - kS : 0;
      for (uint32_t k = first; k < issued; ++k) wait_bar(&fullB[k % kS], (k / kS) & 1, nullptr, nullptr);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer: the whole warp walks the loop (so descriptors stay in
    // uniform registers) and one elected lane issues each instruction ------
    Ring r;
    uint32_t tiles = 0;
    bool polled = false;  // the current ring position is known to be ready
    const uint64_t bdesc0 = smem_desc(tma::smem_u32(B));
    const uint32_t bstep = g.bbytes >> 4;  // descriptor start-address units per B atom
    for (Units w(u0, u1, g.T); w.more(); w.next(), ++tiles) {
      int kc_lo, kc_hi;
      k_range(g, w.t, kc_lo, kc_hi);
      const int ab = tiles & (g.nacc - 1);
      const uint32_t ause = g.nacc == 2 ? tiles >> 1 : tiles;
      // the epilogue must have drained this accumulator
      bool okf = ause == 0 || wait_bar(&accfree[ab], (ause - 1) & 1, timeouts, abortp);
      if (!__all_sync(0xffffffffu, okf)) *abortp = 1;
      tc_fence_after();
      const uint32_t dt = tmem + ab * g.acc_cols;
      for (int kc = kc_lo; kc < kc_hi; ++kc, r.next()) {
        // the stage's copy and block were polled right after the previous
        // step's MMAs went out; wait only if one of them was not complete
        bool ok = true;
        if (!polled)
          ok = !*abortp && wait_bar(&fullB[r.s], r.ph, timeouts, abortp) &&
               wait_bar(&afull[r.s], r.ph, timeouts, abortp);
        if (!__all_sync(0xffffffffu, ok)) { *abortp = 1; polled = false; continue; }
        tc_fence_after();
        const uint64_t bd = bdesc0 + (uint64_t)(r.s * kAtoms * bstep);
        const uint32_t at = tmem + g.acol + 32 * kAtoms * r.s;
        if (elect_one()) {
          // per atom: four K=16 slices, 8 TMEM columns / 32 bytes apart
#pragma unroll
          for (int a = 0; a < kAtoms; ++a) {
            mma_f16_ts(dt, at + 32 * a, bd + a * bstep, g.idesc, (kc > kc_lo || a > 0) ? 1u : 0u);
            mma_f16_ts(dt, at + 32 * a + 8, bd + a * bstep + 2, g.idesc, 1u);
            mma_f16_ts(dt, at + 32 * a + 16, bd + a * bstep + 4, g.idesc, 1u);
            mma_f16_ts(dt, at + 32 * a + 24, bd + a * bstep + 6, g.idesc, 1u);
          }
          mma_commit(&freeS[r.s]);
        }
        __syncwarp();
        // poll the next ring position now (its latency overlaps the loop)
        Ring nx = r;
        nx.next();
        const bool pb = tma::mbar_try_wait(&fullB[nx.s], nx.ph);
        const bool pa = tma::mbar_try_wait(&afull[nx.s], nx.ph);
        polled = pb && pa;
      }
      if (elect_one()) mma_commit(&accfull[ab]);
      __syncwarp();
    }
    // every MMA must be done before the tensor memory is freed
    if (elect_one()) mma_commit(&done);
    __syncwarp();
    wait_bar(&done, 0, nullptr, nullptr);
    __syncwarp();
  } else if (warp >= kEpiWarp0) {
    // ---- epilogue: warp 8+q reads lanes 32q..32q+31 ------------------------
    const int q = warp - kEpiWarp0;
    const int m = q * 32 + lane;
    const uint32_t tlane = tmem + ((uint32_t)(q * 32) << 16);
    const int64_t plane = (int64_t)g.Ho * g.Wo;
    const int64_t nstride = g.out_ctot * plane;
    uint32_t tiles = 0;
    for (Units w(u0, u1, g.T); w.more(); w.next(), ++tiles) {
      const int64_t c = w.c;
      const int t = w.t;
      const int ab = tiles & (g.nacc - 1);
      const uint32_t ause = g.nacc == 2 ? tiles >> 1 : tiles;
      bool ok = !*abortp && wait_bar(&accfull[ab], ause & 1, timeouts, abortp, kSleepNs);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc_fence_after();
        const float bv = bias ? ld(bias + c) : 0.f;
        const int f = t * kM + m;
        const bool mvalid = f < plane;
        T* o0 = y + (g.out_off + c) * plane + f;
        for (int n0 = 0; n0 < g.nb; n0 += 16) {
          float v[16];
          tmem_ld16(tlane + ab * g.acc_cols + n0, v);
          if (mvalid) {
            T* o = o0 + (int64_t)n0 * nstride;
#pragma unroll
            for (int i = 0; i < 16; ++i, o += nstride) {
              if (n0 + i < g.N) {
                const float val = v[i] + bv;
                *o = from_f<T>(accumulate_out ? val + ld_rw(o) : val);
              }
            }
          }
        }
      } else {
        *abortp = 1;
      }
      tc_fence_before();
      mbar_arrive(&accfree[ab]);
    }
  } else {
    // ---- builders ----------------------------------------------------------
    const int quarter = warp & 3, half = warp >> 2;
    const int m = quarter * 32 + lane;  // row of the tile = TMEM lane
    const uint32_t tlane = tmem + ((uint32_t)(quarter * 32) << 16) + g.acol + 32 * half;
    Ring r;
    int64_t cur_c = -1;
    for (Units w(u0, u1, g.T); w.more(); w.next()) {
      const int64_t c = w.c;
      const int t = w.t;
      if (c != cur_c) {
        // eight copies of the padded filter rows, copy s shifted left by s:
        // SC[s][dy][i] = fr(dy, i + s), fr(dy, j) = w'[dy][j - (Wo - 1 - pw)].
        // One warp per (s, dy) row. Every builder has finished the previous
        // channel's steps here.
        builders_sync();
        const T* wc = w_ + c * g.kh * g.kw;
        for (int row = warp; row < 8 * g.kh; row += kBuilders / 32) {
          const int s = row / g.kh, dy = row - s * g.kh;
          const T* wrow = g.flip ? wc + (g.kh - 1 - dy) * g.kw : wc + dy * g.kw;
          T* dst = SC + (size_t)(s * g.kh + dy) * g.L;
          const int b0 = s - (g.Wo - 1 - g.pw);  // filter column of element 0
          for (int i = lane; i < g.L; i += 32) {
            const int b = i + b0;
            float v = 0.f;
            if (b >= 0 && b < g.kw) v = ld(wrow + (g.flip ? g.kw - 1 - b : b));
            dst[i] = from_f<T>(v);
          }
        }
        builders_sync();
        cur_c = c;
      }
      int kc_lo, kc_hi;
      k_range(g, t, kc_lo, kc_hi);
      // this thread's row of the tile: output position f (rows past the plane
      // get an out-of-range filter row, i.e. zeros)
      const int f = t * kM + m;
      const bool mvalid = f < g.Ho * g.Wo;
      const int oh = mvalid ? f / g.Wo : -(1 << 20), ow = mvalid ? f - oh * g.Wo : 0;
      const int j0 = g.Wo - 1 - ow;
      const T* rowsrc = SC + (size_t)(j0 & 7) * g.kh * g.L + (j0 & ~7);
      // first piece of this thread's atom: position kc_lo*kKs + 64*half
      int gpos = kc_lo * kKs + kAtom * half;
      int ih0 = gpos / g.Wi, iw0 = gpos - ih0 * g.Wi;
      for (int kc = kc_lo; kc < kc_hi; ++kc, r.next()) {
        if (r.wrapped && !*abortp && !wait_bar(&freeS[r.s], r.ph ^ 1, timeouts, abortp, kSleepNs)) *abortp = 1;
        tc_fence_after();
        // 8 pieces of 8 input positions: kc*kKs + 64*half + 8j. Positions
        // past the plane meet zero-filled B rows, so their taps do not matter.
        int ih = ih0, iw = iw0;
        uint32_t v32[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int dy = ih - oh + g.ph;
          uint4 v = make_uint4(0, 0, 0, 0);
          if ((unsigned)dy < (unsigned)g.kh) v = *reinterpret_cast<const uint4*>(rowsrc + dy * g.L + iw);
          v32[4 * j] = v.x;
          v32[4 * j + 1] = v.y;
          v32[4 * j + 2] = v.z;
          v32[4 * j + 3] = v.w;
          iw += 8;
          if (iw == g.Wi) { iw = 0; ++ih; }
        }
        tmem_st32(tlane + 32 * kAtoms * r.s, v32);
        tc_fence_before();
        mbar_arrive(&afull[r.s]);
        // advance the first piece by one K step
        iw0 += kKs;
        while (iw0 >= g.Wi) { iw0 -= g.Wi; ++ih0; }
      }
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
  return 1024 + (size_t)S * nb * 128 + (size_t)8 * kh * L * 2;
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

bool fits(const Conv& c, const Geo& q) {
  return smem_bytes(kS * kAtoms, tile::round_up(c.N, 16), c.kh, row_len(q.Wi, q.Wo)) <= 227 * 1024;
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
  if (!fits(c, q)) return cudaErrorInvalidConfiguration;
  // tensor memory: one or two fp32 accumulators (nb columns each), then the
  // A stages (32 columns each)
  g.acc_cols = tile::round_up(g.nb, 32);
  g.nacc = 2 * g.acc_cols + 32 * kAtoms * kS <= 512 ? 2 : 1;
  g.acol = g.nacc * g.acc_cols;
  g.ncols = 32;
  while (g.ncols < g.acol + 32 * kAtoms * kS) g.ncols *= 2;
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
                            (uint32_t)kAtom, 1, (uint32_t)g.nb))
    return cudaErrorInvalidValue;
  size_t smem = smem_bytes(kS * kAtoms, g.nb, g.kh, g.L);
  auto kern = ibgemm_kernel<T>;
  cudaError_t e;
  int dev = 0, sms = 0, occ = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  // CTAs resident per SM, from the kernel's registers and shared memory
  // (computed here: the runtime's occupancy query under-reports it for this
  // kernel). Resident CTAs must never need more than the 512 tensor-memory
  // columns: grow the shared-memory request until few enough fit.
  cudaFuncAttributes fa{};
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  int smem_sm = 0, regs_sm = 0, thr_sm = 0;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) != cudaSuccess) return e;
  const int regs_cta = (kThreads / 32) * ((fa.numRegs * 32 + 255) / 256 * 256);
  const int by_regs = regs_sm / regs_cta, by_thr = thr_sm / kThreads;
  const int tmem_cap = 512 / g.ncols;
  for (;;) {
    const int by_smem = smem_sm / (int)(smem + fa.sharedSizeBytes + 1024);
    occ = by_regs < by_thr ? by_regs : by_thr;
    if (by_smem < occ) occ = by_smem;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    if (occ <= tmem_cap) break;
    smem += 8 * 1024;
  }
  // opt in explicitly: the static shared memory (1 KB) counts against the
  // default 48 KB as well
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
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
  return fits(c, q);
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
