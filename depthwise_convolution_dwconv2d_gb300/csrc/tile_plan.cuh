// Host-side planning of a single-branch tile (shared by the forward and
// stride-1 grad-input kernels).
#pragma once

#include <type_traits>

#include "tile.cuh"
#include "tma.cuh"

namespace dwconv {
namespace tile {

struct Cfg {
  int ppc;          // planes per unit
  int th, nbands;   // output rows per band, bands per plane
  int tr, pitch;    // tile rows / row pitch (elements)
  int rb, cb;       // item grid: row blocks, column blocks
  int ntile;        // staged planes per plane of the unit (1, or m)
  int tile_elems;   // elements per staged plane
  int stage_elems;  // elements per stage
  int mode, ix0;    // copy mode, tile origin column
  int cshift;       // added to each thread's window start column
  int vec_out;
  int tab_floats;   // per-stage side table (filters, bias, plane offsets), floats
  int tab_off64;    // float offset of the 64-bit plane-offset table (even)
  int64_t groups;
  FastDiv trdiv, d_item, d_rb, d_cbq, d_bands;
  uint32_t tma_bytes;  // bytes one stage's tensor copy delivers
  int seg;             // dense staging: elements per plane segment
  int stg_elems;       // dense staging: elements per stage (0 otherwise)
  int balanced;        // equal contiguous plane shares per CTA (see Sched)
  int contig;          // dense staging: a stage's planes are one contiguous run
};


inline bool alignedn(const void* p, int n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Plan a tile for the stencil
//   out[oy][ox] = sum w'[a][b] in[oy*S - ph + a*D][ox*S - pw + b*D]
// with Hin x Win input planes and Hout x Wout output planes. ntile planes are
// staged per plane of a unit; mult output planes are produced per staged
// group. *dl receives the compile-time window offset the kernel needs.
// tma_group: for TMA staging a unit's planes must not straddle a multiple
// of tma_group planes (0: no constraint). *map receives the tensor map when
// TMA staging is chosen.
template <typename T, int K, int S, int D, int R, int V>
bool plan_tile(int64_t nplanes, int ntile, int mult, int64_t Hin, int64_t Win, int64_t Hout,
               int64_t Wout, int pw, const void* in_base, bool out_vec_ok, Cfg* out, int* dl,
               int64_t tma_group, int64_t tma_planes, CUtensorMap* map) {
  constexpr int Q = Geo<K, S, D>::Q, QS = Q * S;
  constexpr int WN = (V - 1) * QS + (K - 1) * D + 1;
  constexpr int ES = sizeof(T);
  Cfg g{};
  int shift = 0;
  g.mode = pick_mode<T>(in_base, Win, -pw, &g.ix0, &shift);
  g.cb = (int)((Wout + (int64_t)Q * V - 1) / ((int64_t)Q * V));
  int64_t need;
  if (Q == 1) {
    *dl = shift % 4;
    g.cshift = shift - *dl;
    const int W4 = (*dl + WN + 3) / 4 * 4;
    need = (int64_t)(g.cb - 1) * V * S + g.cshift + W4;
  } else {
    *dl = 0;
    g.cshift = shift;
    const int64_t owb = (int64_t)(g.cb - 1) * Q * V + Q - 1;
    need = owb * S + shift + WN;
  }
  g.pitch = round_up(need, 16 / ES > 4 ? 16 / ES : 4);
  const int QR = Q * R;
  auto tr_of = [&](int64_t th) { return (th - 1) * S + (int64_t)(K - 1) * D + 1; };
  auto bytes_of = [&](int64_t th) { return tr_of(th) * g.pitch * ES * ntile; };
  const int64_t target = 32 * 1024;  // bytes per stage and plane group
  int64_t th = (Hout + QR - 1) / QR * QR;
  if (bytes_of(th) > target) {
    th = (target / ((int64_t)g.pitch * ES * ntile) - (int64_t)(K - 1) * D - 1) / S + 1;
    th = th / QR * QR;
    if (th < QR) th = QR;
    if (bytes_of(th) > 48 * 1024) return false;
  }
  g.th = (int)th;
  g.rb = (int)(th / QR);
  g.nbands = (int)((Hout + th - 1) / th);
  g.tr = (int)tr_of(th);
  g.ntile = ntile;
  g.tile_elems = g.tr * g.pitch;
  const int64_t items = (int64_t)mult * g.rb * g.cb * Q * Q;
  int64_t ppc = 1;
  if (g.nbands == 1) {
    ppc = (2 * kNT + items - 1) / items;
    const int64_t cap = target / bytes_of(th);
    if (ppc > cap) ppc = cap;
    if (ppc < 1) ppc = 1;
  }
  // dense staging of whole planes when the rows are not 16-byte multiples
  // but the plane bases are (planes of 16-byte multiples), and a plane is
  // one band
  const bool dense_ok = (g.mode == kCopy4 || g.mode == kCopySync) && g.nbands == 1 &&
                        (reinterpret_cast<uintptr_t>(in_base) % 16) == 0;
  if (dense_ok) {
    const int seg = dense_seg<T>(Hin * Win);
    const int64_t per = (int64_t)seg * ntile * ES;  // dense planes are read in place
    int64_t dppc = (2 * kNT + items - 1) / items;
    const int64_t dcap = target / per;
    if (dppc > dcap) dppc = dcap;
    if (dppc >= 1) {
      g.mode = kCopyDense;
      g.seg = seg;
      ppc = dppc;
      // plane groups of a unit never straddle samples (staged planes are
      // addressed per plane, so this only keeps units uniform)
    }
  }
  // TMA staging when the rows allow 16-byte copies and the box fits
  bool tma = g.mode == kCopy16 && g.pitch <= 256 && g.tr <= 256 && ppc * ntile <= 256;
  if (tma && tma_group > 0) {
    while (ppc > 1 && tma_group % ppc != 0) --ppc;  // units never straddle a group
  }
  if (tma) {
    tma = tma::encode_3d(map, in_base, sizeof(T) == 4 ? DWCONV_F32 : (std::is_same<T, __half>::value ? DWCONV_F16 : DWCONV_BF16),
                         (uint64_t)Win, (uint64_t)Hin, (uint64_t)tma_planes, (uint32_t)g.pitch,
                         (uint32_t)g.tr, (uint32_t)(ppc * ntile));
  }
  if (tma) g.mode = kCopyTMA;
  g.ppc = (int)ppc;
  g.groups = (nplanes + ppc - 1) / ppc;
  g.balanced = g.nbands == 1 && g.mode != kCopyTMA;
  g.stage_elems = g.mode == kCopyDense ? 0 : stage_round((int64_t)g.ppc * ntile * g.tile_elems, ES);
  g.tma_bytes = (uint32_t)((int64_t)g.ppc * ntile * g.tile_elems * ES);
  g.stg_elems = g.mode == kCopyDense ? stage_round((int64_t)g.ppc * ntile * g.seg, ES) : 0;
  // side table: K*K filter taps per staged plane (per output plane for the
  // forward: mult * ppc of them), a bias, an epilogue scale and shift and a
  // 64-bit offset each
  const int ntab = g.ppc * (ntile > mult ? ntile : mult);
  g.tab_off64 = round_up((int64_t)ntab * (K * K + 3), 2);
  g.tab_floats = round_up(g.tab_off64 + 2 * (int64_t)ntab, 4);
  g.vec_out = out_vec_ok;
  g.trdiv = FastDiv((uint32_t)g.tr);
  g.d_item = FastDiv((uint32_t)(g.rb * g.cb * Q * Q));
  g.d_rb = FastDiv((uint32_t)(g.cb * Q * Q));
  g.d_cbq = FastDiv((uint32_t)(g.cb * Q));
  g.d_bands = FastDiv((uint32_t)g.nbands);
  *out = g;
  return true;
}

}  // namespace tile
}  // namespace dwconv
