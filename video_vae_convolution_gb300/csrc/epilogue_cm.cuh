// Epilogue of the channel-major convolution kernel: the post-operation contract
// of the cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm + SiLU"
// (section "Operation Contract", bias / residual / residual-bias part; every
// B() is an explicit round-to-nearest-even fp32 -> bf16 conversion), applied to
// a 32-channel x 32-pixel block of the accumulator.
//
// A warp loads its block from TMEM (thread = channel, registers = pixels),
// stages it in shared memory, and then each thread handles units of 8 values
// that are contiguous in the output: 8 channels of one pixel for NDHWC output
// (16-byte loads and stores, coalesced across the warp) or 8 pixels of one
// channel for NCDHW output.
//
// Layers with little reduction work per output element (narrow input, 96
// channels) are bound by this code, so the per-unit work is kept short: one
// division per block for the pixel positions, the thread's bias values held in
// registers for the whole tile, 16-byte shared-memory reads.
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "internal.h"

namespace vvc {

struct CmEpi {
  unsigned flags;
  int Cout, Do, Ho, Wo, Hy, Wy;
  bool ndhwc, pad, split;
  uint16_t* y;
  const uint16_t* res;
  uint16_t* val;
  uint16_t* conv;
  float* part;
  const float* bias;
  const float* rbias;
  const float* gamma;
  float sqrt_c;
  long long M_total;
  bool halo;              // y is haloed (NDHWC): addresses and extras from *ep
  const EpiParams* ep;    // the launch's epilogue parameters (kernel parameter space)
  bool up2;               // x2 upsampled input: y is [N, Do, 2 Ho, 2 Wo, Cout]
};

struct CmTile {
  int nb, od, split;
  int w0, h0, tw, npix;
  // flat: tile pixel n is flattened position w0 + n of the plane (row pitch `pitch` = W);
  // otherwise pixel n is output row h0 + n / pitch, column w0 + n % pitch, and only
  // columns n % pitch < tw belong to the tile (the rest are halo rows of a run)
  int flat, pitch;
  // the same as a row/column split of q = q0 + n by pitch: output row hoff + q / pitch,
  // column woff + q % pitch, in the tile while the column index is below jlim
  int q0, hoff, woff, jlim;
  // vrows > 0: the tile runs over the flattened volume; its row index counts rows of
  // the input volume, frame = row / vrows (the input height), row in frame = the rest
  int vrows;
  int cls;  // parity class of an x2 upsampled input (output row 2 h + cls / 2, column
            // 2 w + cls % 2)
};

// Element offset of channel c of tile output (nd = n * Do + d, h, w) in y and conv_out
// when the input is x2 upsampled: the class's pixel of the [2 Ho, 2 Wo] output.
__device__ __forceinline__ long long cm_up2_offset(const CmEpi& E, const CmTile& t, long long nd,
                                                   int h, int w, int c) {
  return ((nd * (2LL * E.Ho) + 2 * h + (t.cls >> 1)) * (2LL * E.Wo) + 2 * w + (t.cls & 1)) *
             E.Cout + c;
}

// Output frame and row of tile row index hv (see CmTile::vrows).
__device__ __forceinline__ void cm_frame_row(const CmTile& t, int hv, int& d, int& h) {
  if (t.vrows) {
    d = hv / t.vrows;
    h = hv - d * t.vrows;
  } else {
    d = t.od;
    h = hv;
  }
}

// Per-warp staging block: 32 rows (pixels) of 32 channels, fp32.  Rows are
// kStageVec floats apart where a thread reads 8 channels of a pixel as two
// 16-byte words, kStageScalar floats apart where threads read along a row.
constexpr int kStageVec = 36;
constexpr int kStageScalar = 33;
constexpr int kStageFloats = 32 * kStageVec;  // per warp

// The 8 output channels [c0, c0 + cnt) of one epilogue thread in the NDHWC units
// (lanes 4k + g share a pixel; g = lane & 3), with their bias and residual bias.
struct CmChan {
  int c0, cnt;
  float b[8], rb[8];
  float bc;  // bias of the thread's own TMEM channel (bulk-store blocks)
};

__device__ __forceinline__ CmChan cm_chan(const CmEpi& E, int cw, int lane) {
  CmChan c;
  c.c0 = cw + 8 * (lane & 3);
  c.cnt = min(8, E.Cout - c.c0);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const bool in = e < c.cnt;
    c.b[e] = ((E.flags & EPI_BIAS) && in) ? __ldg(E.bias + c.c0 + e) : 0.0f;
    c.rb[e] = ((E.flags & EPI_RESIDUAL_BIAS) && in) ? __ldg(E.rbias + c.c0 + e) : 0.0f;
  }
  c.bc = ((E.flags & EPI_BIAS) && cw + lane < E.Cout) ? __ldg(E.bias + cw + lane) : 0.0f;
  return c;
}

// Row index (see CmTile::vrows) and column of tile pixel j0 + pl from the block
// origin (ib, jb) of pixel j0; true when the pixel belongs to the tile.
__device__ __forceinline__ bool cm_unit_pos_v(const CmTile& t, int ib, int jb, int j0, int pl,
                                              int& hv, int& w) {
  int i = ib, j = jb + pl;
  while (j >= t.pitch) {
    j -= t.pitch;
    ++i;
  }
  hv = t.hoff + i;
  w = t.woff + j;
  return j < t.jlim && j0 + pl < t.npix;
}

// Row / column of tile pixel j0 + pl from the block origin (ib, jb) of pixel j0;
// true when the pixel belongs to the tile and lies inside the output.
__device__ __forceinline__ bool cm_unit_pos(const CmEpi& E, const CmTile& t, int ib, int jb,
                                            int j0, int pl, int& h, int& w) {
  int i = ib, j = jb + pl;
  while (j >= t.pitch) {
    j -= t.pitch;
    ++i;
  }
  h = t.hoff + i;
  w = t.woff + j;
  return j < t.jlim && j0 + pl < t.npix && h < E.Ho && w < E.Wo;
}

// value = B(B(B(acc) + bias) + B(res + rbias)) for the 8 channels of a unit;
// conv bits kept for the debug store.  `res_at(e)` gives the residual element.
template <class Res>
__device__ __forceinline__ void cm_value8(const CmEpi& E, const CmChan& ch, const float (&a)[8],
                                          uint16_t (&cb)[8], float (&v)[8], Res&& res8) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    cb[e] = bf16_bits(a[e]);
    v[e] = bf16_val(cb[e]);
  }
  if (E.flags & EPI_BIAS) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = round_bf16(__fadd_rn(v[e], ch.b[e]));
  }
  if (E.flags & EPI_RESIDUAL) {
    float sk[8];
    res8(sk);
    if (E.flags & EPI_RESIDUAL_BIAS) {
#pragma unroll
      for (int e = 0; e < 8; ++e) sk[e] = round_bf16(__fadd_rn(sk[e], ch.rb[e]));
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = round_bf16(__fadd_rn(v[e], sk[e]));
  }
}

// Output coordinates of tile pixel n; false when n is not one of the tile's pixels.
// The caller still checks h < Ho and w < Wo.
__device__ __forceinline__ bool cm_pixel(const CmTile& t, int n, int& h, int& w) {
  if (t.flat) {
    const int q = t.w0 + n;
    h = q / t.pitch;
    w = q - h * t.pitch;
    return true;
  }
  const int i = n / t.pitch;
  const int j = n - i * t.pitch;
  h = t.h0 + i;
  w = t.w0 + j;
  return j < t.tw;
}

// Whether tile pixels [n, n + len) lie on one output row at consecutive w.
__device__ __forceinline__ bool cm_same_row(const CmTile& t, int n, int len) {
  if (t.flat) return ((t.w0 + n) % t.pitch) + len <= t.pitch;
  return (n % t.pitch) + len <= t.tw;
}

__device__ __forceinline__ uint4 pack8(const uint16_t (&v)[8]) {
  uint4 u;
  u.x = v[0] | (uint32_t(v[1]) << 16);
  u.y = v[2] | (uint32_t(v[3]) << 16);
  u.z = v[4] | (uint32_t(v[5]) << 16);
  u.w = v[6] | (uint32_t(v[7]) << 16);
  return u;
}

__device__ __forceinline__ void unpack8(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Two fp32 values -> packed bf16x2 (round to nearest even; lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ float bf16x2_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16x2_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// NDHWC output (or split partial sums) for one 32-channel x 32-pixel block staged
// at st (rows kStageVec apart): unit = (pixel, the thread's 8 channels).
__device__ __forceinline__ void cm_block_ndhwc(const CmEpi& E, const CmTile& t, const float* st,
                                               int lane, const CmChan& ch, int j0) {
  const int q = t.q0 + j0;
  const int ib = q / t.pitch;
  const int jb = q - ib * t.pitch;
  const bool vec = (ch.cnt == 8) && ((E.Cout & 7) == 0);
  const int g = lane & 3;
  int fd, hrow;  // frame and row of the block's first pixel
  cm_frame_row(t, t.hoff + ib, fd, hrow);
  // Fast path: the block's 32 pixels are consecutive pixels of one output row, all
  // inside the output, and the thread's 8 channels are a full 16-byte group.  One
  // base address per block; values converted two at a time.
  if (vec && !E.split && !E.pad && jb + 31 < t.jlim && jb + 31 < t.pitch && j0 + 31 < t.npix &&
      hrow < E.Ho && fd < E.Do && t.woff + jb + 31 < E.Wo) {
    const long long nd = (long long)t.nb * E.Do + fd;
    const int wcol = t.woff + jb + (lane >> 2);
    const long long o0 = ((nd * E.Ho + hrow) * E.Wo + wcol) * E.Cout + ch.c0;
    // y offset of the thread's first pixel (a haloed y has its own geometry)
    const long long oy0 = E.halo  ? halo_offset(*E.ep, t.nb, fd, hrow, wcol, ch.c0)
                          : E.up2 ? cm_up2_offset(E, t, nd, hrow, wcol, ch.c0)
                                  : o0;
    const long long step = 8LL * E.Cout;  // the thread's next pixel is 8 pixels on
    const long long ystep = E.up2 ? 2 * step : step;  // (every other output pixel)
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int pl = 8 * k + (lane >> 2);
      const long long o = o0 + k * step;
      const float4 lo = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g);
      const float4 hi = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g + 4);
      uint4 cb;  // B(conv)
      cb.x = pack_bf16x2(lo.x, lo.y);
      cb.y = pack_bf16x2(lo.z, lo.w);
      cb.z = pack_bf16x2(hi.x, hi.y);
      cb.w = pack_bf16x2(hi.z, hi.w);
      uint4 v = cb;
      if (E.flags & EPI_BIAS) {
        v.x = pack_bf16x2(__fadd_rn(bf16x2_lo(v.x), ch.b[0]), __fadd_rn(bf16x2_hi(v.x), ch.b[1]));
        v.y = pack_bf16x2(__fadd_rn(bf16x2_lo(v.y), ch.b[2]), __fadd_rn(bf16x2_hi(v.y), ch.b[3]));
        v.z = pack_bf16x2(__fadd_rn(bf16x2_lo(v.z), ch.b[4]), __fadd_rn(bf16x2_hi(v.z), ch.b[5]));
        v.w = pack_bf16x2(__fadd_rn(bf16x2_lo(v.w), ch.b[6]), __fadd_rn(bf16x2_hi(v.w), ch.b[7]));
      }
      if (E.flags & EPI_RESIDUAL) {
        uint4 sk = __ldg(reinterpret_cast<const uint4*>(E.res + o));
        if (E.flags & EPI_RESIDUAL_BIAS) {
          sk.x = pack_bf16x2(__fadd_rn(bf16x2_lo(sk.x), ch.rb[0]),
                             __fadd_rn(bf16x2_hi(sk.x), ch.rb[1]));
          sk.y = pack_bf16x2(__fadd_rn(bf16x2_lo(sk.y), ch.rb[2]),
                             __fadd_rn(bf16x2_hi(sk.y), ch.rb[3]));
          sk.z = pack_bf16x2(__fadd_rn(bf16x2_lo(sk.z), ch.rb[4]),
                             __fadd_rn(bf16x2_hi(sk.z), ch.rb[5]));
          sk.w = pack_bf16x2(__fadd_rn(bf16x2_lo(sk.w), ch.rb[6]),
                             __fadd_rn(bf16x2_hi(sk.w), ch.rb[7]));
        }
        v.x = pack_bf16x2(__fadd_rn(bf16x2_lo(v.x), bf16x2_lo(sk.x)),
                          __fadd_rn(bf16x2_hi(v.x), bf16x2_hi(sk.x)));
        v.y = pack_bf16x2(__fadd_rn(bf16x2_lo(v.y), bf16x2_lo(sk.y)),
                          __fadd_rn(bf16x2_hi(v.y), bf16x2_hi(sk.y)));
        v.z = pack_bf16x2(__fadd_rn(bf16x2_lo(v.z), bf16x2_lo(sk.z)),
                          __fadd_rn(bf16x2_hi(v.z), bf16x2_hi(sk.z)));
        v.w = pack_bf16x2(__fadd_rn(bf16x2_lo(v.w), bf16x2_lo(sk.w)),
                          __fadd_rn(bf16x2_hi(v.w), bf16x2_hi(sk.w)));
      }
      *reinterpret_cast<uint4*>(E.y + oy0 + k * ystep) = v;
      if (E.flags & EPI_SAVE_VALUE) *reinterpret_cast<uint4*>(E.val + o) = v;
      if (E.flags & EPI_DEBUG_STORE_CONV)
        *reinterpret_cast<uint4*>(E.conv + (E.up2 ? oy0 + k * ystep : o)) = cb;
      if (E.halo) {
        halo_extras(*E.ep, t.nb, fd, hrow, wcol + 8 * k, ch.c0, [&](long long off, bool zero) {
          *reinterpret_cast<uint4*>(E.y + off) = zero ? make_uint4(0u, 0u, 0u, 0u) : v;
        });
      }
    }
    return;
  }
  for (int k = 0; k < 4; ++k) {
    const int pl = 8 * k + (lane >> 2);
    int hv, h, w, d;
    if (ch.cnt <= 0 || !cm_unit_pos_v(t, ib, jb, j0, pl, hv, w)) continue;
    cm_frame_row(t, hv, d, h);
    if (h >= E.Ho || w >= E.Wo || d >= E.Do) continue;
    const long long nd = (long long)t.nb * E.Do + d;
    float a[8];
    {
      const float4 lo = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g);
      const float4 hi = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g + 4);
      a[0] = lo.x; a[1] = lo.y; a[2] = lo.z; a[3] = lo.w;
      a[4] = hi.x; a[5] = hi.y; a[6] = hi.z; a[7] = hi.w;
    }
    const long long pix = (nd * E.Ho + h) * E.Wo + w;
    if (E.split) {
      float* dst = E.part + ((long long)t.split * E.M_total + pix) * E.Cout + ch.c0;
      if (vec) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(a[0], a[1], a[2], a[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(a[4], a[5], a[6], a[7]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (e < ch.cnt) dst[e] = a[e];
      }
      continue;
    }
    const long long ou = pix * E.Cout + ch.c0;
    uint16_t cb[8];
    float v[8];
    cm_value8(E, ch, a, cb, v, [&](float (&sk)[8]) {
      if (vec) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(E.res + ou)), sk);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) sk[e] = (e < ch.cnt) ? bf16_val(E.res[ou + e]) : 0.0f;
      }
    });
    uint16_t vb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) vb[e] = bf16_bits(v[e]);
    const long long yo = E.halo  ? halo_offset(*E.ep, t.nb, d, h, w, ch.c0)
                         : E.up2 ? cm_up2_offset(E, t, nd, h, w, ch.c0)
                                 : ((nd * E.Hy + h) * E.Wy + w) * E.Cout + ch.c0;
    if (E.up2) {
      // x2 upsampled input (Cout % 8 == 0; no residual or saved value): y and the
      // debug conv store take the class's output pixel
      reinterpret_cast<uint4*>(E.y + yo)[0] = pack8(vb);
      if (E.flags & EPI_DEBUG_STORE_CONV) reinterpret_cast<uint4*>(E.conv + yo)[0] = pack8(cb);
      continue;
    }
    if (E.halo) {
      // (a haloed y has Cout % 8 == 0, so the thread's 8 channels are one 16-byte group)
      const uint4 pv = pack8(vb);
      reinterpret_cast<uint4*>(E.y + yo)[0] = pv;
      if (E.flags & EPI_SAVE_VALUE) reinterpret_cast<uint4*>(E.val + ou)[0] = pv;
      if (E.flags & EPI_DEBUG_STORE_CONV) reinterpret_cast<uint4*>(E.conv + ou)[0] = pack8(cb);
      halo_extras(*E.ep, t.nb, d, h, w, ch.c0, [&](long long off, bool zero) {
        *reinterpret_cast<uint4*>(E.y + off) = zero ? make_uint4(0u, 0u, 0u, 0u) : pv;
      });
      continue;
    }
    if (vec) {
      const uint4 pv = pack8(vb);
      reinterpret_cast<uint4*>(E.y + yo)[0] = pv;
      if (E.flags & EPI_SAVE_VALUE) reinterpret_cast<uint4*>(E.val + ou)[0] = pv;
      if (E.flags & EPI_DEBUG_STORE_CONV) reinterpret_cast<uint4*>(E.conv + ou)[0] = pack8(cb);
      if (E.pad) {
        const uint4 z = make_uint4(0, 0, 0, 0);
        const long long sw_ = E.Cout, sh_ = (long long)E.Wy * E.Cout;
        if (w == E.Wo - 1) reinterpret_cast<uint4*>(E.y + yo + sw_)[0] = z;
        if (h == E.Ho - 1) reinterpret_cast<uint4*>(E.y + yo + sh_)[0] = z;
        if (w == E.Wo - 1 && h == E.Ho - 1) reinterpret_cast<uint4*>(E.y + yo + sh_ + sw_)[0] = z;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e >= ch.cnt) continue;
        E.y[yo + e] = vb[e];
        if (E.flags & EPI_SAVE_VALUE) E.val[ou + e] = vb[e];
        if (E.flags & EPI_DEBUG_STORE_CONV) E.conv[ou + e] = cb[e];
        if (E.pad) {
          const long long sw_ = E.Cout, sh_ = (long long)E.Wy * E.Cout;
          if (w == E.Wo - 1) E.y[yo + e + sw_] = 0;
          if (h == E.Ho - 1) E.y[yo + e + sh_] = 0;
          if (w == E.Wo - 1 && h == E.Ho - 1) E.y[yo + e + sh_ + sw_] = 0;
        }
      }
    }
  }
}

// 8 consecutive tile pixels [n0, n0 + 8) of one channel c, NCDHW addressing.
__device__ __forceinline__ void cm_unit_ncdhw(const CmEpi& E, const CmTile& t, int n0, int c,
                                              const float (&a)[8]) {
  if (c >= E.Cout) return;
  const float bias_c = (E.flags & EPI_BIAS) ? __ldg(E.bias + c) : 0.0f;
  const float rb_c = (E.flags & EPI_RESIDUAL_BIAS) ? __ldg(E.rbias + c) : 0.0f;
  const long long ncd = ((long long)t.nb * E.Cout + c) * E.Do + t.od;
  const long long nd = (long long)t.nb * E.Do + t.od;
  int h0, w0;
  cm_pixel(t, n0, h0, w0);
  // fast path: 8 pixels of one output row, all valid, 16-byte aligned
  const bool vec = (n0 + 8 <= t.npix) && (w0 + 8 <= E.Wo) && (h0 < E.Ho) &&
                   cm_same_row(t, n0, 8) && ((w0 & 7) == 0) && ((E.Wo & 7) == 0) &&
                   !E.split && !(E.flags & EPI_DEBUG_STORE_CONV) && !E.pad;
  if (vec) {
    const long long ou = ncd * ((long long)E.Ho * E.Wo) + (long long)h0 * E.Wo + w0;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = round_bf16(a[e]);
      if (E.flags & EPI_BIAS) v[e] = round_bf16(__fadd_rn(v[e], bias_c));
    }
    if (E.flags & EPI_RESIDUAL) {
      float sk[8];
      unpack8(__ldg(reinterpret_cast<const uint4*>(E.res + ou)), sk);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (E.flags & EPI_RESIDUAL_BIAS) sk[e] = round_bf16(__fadd_rn(sk[e], rb_c));
        v[e] = round_bf16(__fadd_rn(v[e], sk[e]));
      }
    }
    uint16_t vb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) vb[e] = bf16_bits(v[e]);
    const uint4 pv = pack8(vb);
    reinterpret_cast<uint4*>(E.y + ou)[0] = pv;  // Hy == Ho, Wy == Wo without the pad
    if (E.flags & EPI_SAVE_VALUE) reinterpret_cast<uint4*>(E.val + ou)[0] = pv;
    return;
  }
  for (int e = 0; e < 8; ++e) {
    int h, w;
    const bool in_tile = cm_pixel(t, n0 + e, h, w);
    if (!in_tile || n0 + e >= t.npix || h >= E.Ho || w >= E.Wo) continue;
    const long long pix = (nd * E.Ho + h) * E.Wo + w;
    if (E.split) {
      E.part[((long long)t.split * E.M_total + pix) * E.Cout + c] = a[e];
      continue;
    }
    const uint16_t cb = bf16_bits(a[e]);
    float v = bf16_val(cb);
    if (E.flags & EPI_BIAS) v = round_bf16(__fadd_rn(v, bias_c));
    const long long ou = ncd * ((long long)E.Ho * E.Wo) + (long long)h * E.Wo + w;
    if (E.flags & EPI_RESIDUAL) {
      float sk = bf16_val(E.res[ou]);
      if (E.flags & EPI_RESIDUAL_BIAS) sk = round_bf16(__fadd_rn(sk, rb_c));
      v = round_bf16(__fadd_rn(v, sk));
    }
    const uint16_t vb = bf16_bits(v);
    if (E.flags & EPI_DEBUG_STORE_CONV) E.conv[pix * E.Cout + c] = cb;
    if (E.flags & EPI_SAVE_VALUE) E.val[ou] = vb;
    const long long yo = ncd * ((long long)E.Hy * E.Wy) + (long long)h * E.Wy + w;
    E.y[yo] = vb;
    if (E.pad) {
      if (w == E.Wo - 1) E.y[yo + 1] = 0;
      if (h == E.Ho - 1) E.y[yo + E.Wy] = 0;
      if (w == E.Wo - 1 && h == E.Ho - 1) E.y[yo + E.Wy + 1] = 0;
    }
  }
}

// One 32-channel x 32-pixel block: r[j] = accumulator of this lane's channel for
// tile pixel j0 + j.  `st` is this warp's staging block (kStageFloats floats).
__device__ __forceinline__ void cm_block(const CmEpi& E, const CmTile& t, float* st, int lane,
                                         int cw, int j0, const uint32_t (&r)[32],
                                         const CmChan& ch) {
  if (E.ndhwc || E.split) {
#pragma unroll
    for (int j = 0; j < 32; ++j) st[j * kStageVec + lane] = __uint_as_float(r[j]);
    __syncwarp();
    cm_block_ndhwc(E, t, st, lane, ch, j0);
  } else {
    float(*stage)[kStageScalar] = reinterpret_cast<float(*)[kStageScalar]>(st);
#pragma unroll
    for (int j = 0; j < 32; ++j) stage[j][lane] = __uint_as_float(r[j]);
    __syncwarp();
    int h0, w0;
    cm_pixel(t, j0, h0, w0);
    // a plain y = B(B(conv) + bias) block goes to the per-pixel loop below even when
    // its row is aligned: one warp-wide 64-byte store per channel plane beats eight
    // 16-byte stores into 32 different planes
    const bool plain = !(E.flags & (EPI_RESIDUAL | EPI_SAVE_VALUE | EPI_DEBUG_STORE_CONV)) &&
                       !E.pad;
    const bool row_aligned =
        !plain && cm_same_row(t, j0, 32) && (w0 & 7) == 0 && (E.Wo & 7) == 0;
    if (row_aligned) {
      // unit = (channel = lane, 8 consecutive pixels): 16-byte stores
      for (int k = 0; k < 4; ++k) {
        float a[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) a[e] = stage[8 * k + e][lane];
        cm_unit_ncdhw(E, t, j0 + 8 * k, cw + lane, a);
      }
    } else {
      // lane = pixel: for each channel, the warp writes 32 consecutive pixels
      const int n = j0 + lane;
      int h, w;
      const bool in_tile = cm_pixel(t, n, h, w);
      const bool pv = in_tile && n < t.npix && h < E.Ho && w < E.Wo;
      const long long plane_o = (long long)E.Ho * E.Wo, plane_y = (long long)E.Hy * E.Wy;
      const long long pix = (((long long)t.nb * E.Do + t.od) * E.Ho + h) * E.Wo + w;
      const int cend = min(32, E.Cout - cw);
      // 8 channels per step: eight independent chains per lane keep the single
      // epilogue warp of each scheduler busy.
      const long long ou0 = ((long long)t.nb * E.Cout + cw) * E.Do * plane_o +
                            (long long)t.od * plane_o + (long long)h * E.Wo + w;
      const long long yo0 = ((long long)t.nb * E.Cout + cw) * E.Do * plane_y +
                            (long long)t.od * plane_y + (long long)h * E.Wy + w;
      const long long cstep_o = (long long)E.Do * plane_o, cstep_y = (long long)E.Do * plane_y;
      if (plain) {
        // y = B(B(conv) + bias): one pointer stepping through the channel planes; the
        // bias of channel cw + cc comes from lane cc, which holds it for its own channel
        const bool bias = (E.flags & EPI_BIAS) != 0;
        uint16_t* yp = E.y + yo0;
#pragma unroll 8
        for (int cc = 0; cc < 32; ++cc) {
          const float bc = __shfl_sync(0xffffffffu, ch.bc, cc);
          if (cc < cend && pv) {
            float v = round_bf16(stage[lane][cc]);
            if (bias) v = __fadd_rn(v, bc);
            *yp = bf16_bits(v);
          }
          yp += cstep_y;
        }
        __syncwarp();  // the staging block is rewritten by the next block
        return;
      }
      for (int cc0 = 0; cc0 < cend; cc0 += 8) {
        float v[8];
        uint16_t cb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          cb[e] = bf16_bits(stage[lane][cc0 + e]);
          v[e] = bf16_val(cb[e]);
        }
        if (!pv) continue;
        if (E.flags & EPI_BIAS) {
#pragma unroll
          for (int e = 0; e < 8; ++e)
            if (cc0 + e < cend) v[e] = round_bf16(__fadd_rn(v[e], __ldg(E.bias + cw + cc0 + e)));
        }
        if (E.flags & EPI_RESIDUAL) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (cc0 + e >= cend) continue;
            float sk = bf16_val(E.res[ou0 + (cc0 + e) * cstep_o]);
            if (E.flags & EPI_RESIDUAL_BIAS)
              sk = round_bf16(__fadd_rn(sk, __ldg(E.rbias + cw + cc0 + e)));
            v[e] = round_bf16(__fadd_rn(v[e], sk));
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (cc0 + e >= cend) continue;
          const uint16_t vb = bf16_bits(v[e]);
          const long long ou = ou0 + (cc0 + e) * cstep_o;
          const long long yo = yo0 + (cc0 + e) * cstep_y;
          if (E.flags & EPI_DEBUG_STORE_CONV) E.conv[pix * E.Cout + cw + cc0 + e] = cb[e];
          if (E.flags & EPI_SAVE_VALUE) E.val[ou] = vb;
          E.y[yo] = vb;
          if (E.pad) {
            if (w == E.Wo - 1) E.y[yo + 1] = 0;
            if (h == E.Ho - 1) E.y[yo + E.Wy] = 0;
            if (w == E.Wo - 1 && h == E.Ho - 1) E.y[yo + E.Wy + 1] = 0;
          }
        }
      }
    }
  }
  __syncwarp();
}

// Halo writes of a bulk-stored NDHWC block (32 pixels of output row hr from column wr,
// channels cw..cw + 31, staged as bf16 [pixel][32] at yt) besides the bulk stores of
// the block and of its reflected rows: zero halo rows beside the row, and the halo
// columns of the block's pixels next to the row ends (in the row and its halo rows).
// bh: halo_bits of the row.  16 bytes a lane.
static __device__ __noinline__ void cm_halo_block(const EpiParams& e, const uint16_t* yt, int lane,
                                           int nb, int od, int hr, int wr, int cw, int bh) {
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  const int part = lane & 3;
  for (int side = 0; side < 2; ++side) {
    const int hb = side ? (bh >> 2) : bh;  // bits of halo row -1 / Ho
    if ((hb & 3) != 3) continue;           // only zero halo rows are written here
    const int hh = side ? e.Ho : -1;
    for (int u = lane; u < 128; u += 32)
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(e.y) +
                                halo_offset(e, nb, od, hh, wr + (u >> 2), cw + 8 * (u & 3))) =
          zero4;
  }
  // halo columns: each W side copies one output column (reflect: 1 and Wo - 2) or
  // borders one (zero: 0 and Wo - 1); lanes 0-3 write that pixel's 32 channels when it
  // lies in this block (the pixels halo_bits marks)
  if (lane >= 4) return;
  uint16_t* y = static_cast<uint16_t*>(e.y);
  const bool zc = e.w_mode != 2;
  for (int cs = 0; cs < 2; ++cs) {
    if (!(cs ? (e.Wy - e.Wo - e.w0 > 0) : (e.w0 > 0))) continue;
    const int j = (cs ? (zc ? e.Wo - 1 : e.Wo - 2) : (zc ? 0 : 1)) - wr;
    if (j < 0 || j >= 32) continue;
    const uint4 val = *reinterpret_cast<const uint4*>(yt + j * 32 + 8 * part);
    const int ww = cs ? e.Wo : -1;
    *reinterpret_cast<uint4*>(y + halo_offset(e, nb, od, hr, ww, cw + 8 * part)) =
        zc ? zero4 : val;
    if (bh & 1)
      *reinterpret_cast<uint4*>(y + halo_offset(e, nb, od, -1, ww, cw + 8 * part)) =
          (zc || (bh & 2)) ? zero4 : val;
    if (bh & 4)
      *reinterpret_cast<uint4*>(y + halo_offset(e, nb, od, e.Ho, ww, cw + 8 * part)) =
          (zc || (bh & 8)) ? zero4 : val;
  }
}

// ---- fused L2 norm over the channel row ---------------------------------------------
//
// The norm needs every output channel of a pixel, while a tile holds 128 of them.
// All channel tiles of one pixel tile therefore run on the same CTA, one after
// the other.  Pass 1 (once per channel tile) turns the accumulators into values
// and keeps them as bf16 in the CTA's scratch rows (row n = tile pixel n, Cs =
// Cout rounded up to 8 channels; the rows are rewritten for every pixel tile, so
// they stay in L2).  After the last channel tile one thread per pixel sums
// value^2 over the row serially in channel order (as the contract's fp32 sum;
// the square of a bf16 value is exact in fp32), and pass 2 normalizes, scales,
// applies gamma and SiLU, and stores y.

// Residual element offset of (pixel (h, w) of the tile's plane, channel c).
__device__ __forceinline__ long long cm_res_offset(const CmEpi& E, const CmTile& t, int h, int w,
                                                   int c) {
  if (E.ndhwc)
    return ((((long long)t.nb * E.Do + t.od) * E.Ho + h) * E.Wo + w) * E.Cout + c;
  return (((long long)t.nb * E.Cout + c) * E.Do + t.od) * ((long long)E.Ho * E.Wo) +
         (long long)h * E.Wo + w;
}

// Pass 1 for one 32-channel x 32-pixel block (r[j] = accumulator of this lane's
// channel cw + lane at tile pixel j0 + j).
__device__ __forceinline__ void cm_norm_pass1(const CmEpi& E, const CmTile& t, float* st, int lane,
                                              int j0, const uint32_t (&r)[32], uint16_t* scr,
                                              int Cs, const CmChan& ch) {
#pragma unroll
  for (int j = 0; j < 32; ++j) st[j * kStageVec + lane] = __uint_as_float(r[j]);
  __syncwarp();
  const int q = t.q0 + j0;
  const int ib = q / t.pitch;
  const int jb = q - ib * t.pitch;
  const int g = lane & 3;
  const bool vec = (ch.cnt == 8) && ((E.Cout & 7) == 0) && E.ndhwc;
  const long long cstep = E.ndhwc ? 1 : (long long)E.Do * E.Ho * E.Wo;
  for (int k = 0; k < 4; ++k) {
    const int pl = 8 * k + (lane >> 2);
    const int n = j0 + pl;
    int h, w;
    if (ch.cnt <= 0 || !cm_unit_pos(E, t, ib, jb, j0, pl, h, w)) continue;
    float a[8];
    {
      const float4 lo = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g);
      const float4 hi = *reinterpret_cast<const float4*>(st + pl * kStageVec + 8 * g + 4);
      a[0] = lo.x; a[1] = lo.y; a[2] = lo.z; a[3] = lo.w;
      a[4] = hi.x; a[5] = hi.y; a[6] = hi.z; a[7] = hi.w;
    }
    uint16_t cb[8], vb[8];
    float v[8];
    cm_value8(E, ch, a, cb, v, [&](float (&sk)[8]) {
      const long long ro = cm_res_offset(E, t, h, w, ch.c0);
      if (vec) {
        unpack8(__ldg(reinterpret_cast<const uint4*>(E.res + ro)), sk);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) sk[e] = (e < ch.cnt) ? bf16_val(E.res[ro + e * cstep]) : 0.0f;
      }
    });
#pragma unroll
    for (int e = 0; e < 8; ++e) vb[e] = (e < ch.cnt) ? bf16_bits(v[e]) : uint16_t(0);
    *reinterpret_cast<uint4*>(scr + (long long)n * Cs + ch.c0) = pack8(vb);
    if (E.flags & EPI_DEBUG_STORE_CONV) {
      const long long pix = (((long long)t.nb * E.Do + t.od) * E.Ho + h) * E.Wo + w;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (e < ch.cnt) E.conv[pix * E.Cout + ch.c0 + e] = cb[e];
    }
  }
  __syncwarp();
}

// den of tile pixel n from its scratch row: serial fp32 sum in channel order.
__device__ __forceinline__ float cm_norm_den(const CmEpi& E, const uint16_t* row) {
  float ss = 0.0f;
  const int full = E.Cout & ~7;
#pragma unroll 2
  for (int c = 0; c < full; c += 8) {
    float v[8];
    unpack8(*reinterpret_cast<const uint4*>(row + c), v);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = __fadd_rn(ss, __fmul_rn(v[e], v[e]));
  }
  for (int c = full; c < E.Cout; ++c) {
    const float v = bf16_val(row[c]);
    ss = __fadd_rn(ss, __fmul_rn(v, v));
  }
  return norm_den(ss);
}

// Pass 2, NDHWC output: units of (tile pixel, 8 channels) over the 256 epilogue
// threads; consecutive threads take consecutive channel groups of a pixel.
__device__ __forceinline__ void cm_norm_pass2_ndhwc(const CmEpi& E, const CmTile& t, int tid,
                                                    int nthreads, int N, const uint16_t* scr,
                                                    int Cs, const float* den) {
  const int G = Cs / 8;
  const int units = N * G;
  const long long nd = (long long)t.nb * E.Do + t.od;
  const bool vec = (E.Cout & 7) == 0;
  for (int u = tid; u < units; u += nthreads) {
    const int n = u / G;
    const int c0 = 8 * (u - n * G);
    int h, w;
    const bool in_tile = cm_pixel(t, n, h, w);
    if (!in_tile || n >= t.npix || h >= E.Ho || w >= E.Wo) continue;
    const int cnt = min(8, E.Cout - c0);
    const uint4 raw = *reinterpret_cast<const uint4*>(scr + (long long)n * Cs + c0);
    float v[8];
    unpack8(raw, v);
    const long long o = ((nd * E.Ho + h) * E.Wo + w) * E.Cout + c0;
    const float dn = den[n];
    uint16_t yb[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float gm = (e < cnt) ? __ldg(E.gamma + c0 + e) : 0.0f;
      yb[e] = bf16_bits(norm_silu1(v[e], dn, E.sqrt_c, gm));
    }
    if (vec) {
      if (E.flags & EPI_SAVE_VALUE) reinterpret_cast<uint4*>(E.val + o)[0] = raw;
      reinterpret_cast<uint4*>(E.y + o)[0] = pack8(yb);
    } else {
      const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
      for (int e = 0; e < cnt; ++e) {
        if (E.flags & EPI_SAVE_VALUE)
          E.val[o + e] = static_cast<uint16_t>((rw[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
        E.y[o + e] = yb[e];
      }
    }
  }
}

// Pass 2, NCDHW output: 32-pixel x 32-channel blocks per warp, transposed in the
// warp's staging block so that each store covers consecutive pixels of a channel.
__device__ __forceinline__ void cm_norm_pass2_ncdhw(const CmEpi& E, const CmTile& t, float* st,
                                                    int lane, int warp_e, int nwarps, int N,
                                                    const uint16_t* scr, int Cs,
                                                    const float* den) {
  float(*stage)[kStageScalar] = reinterpret_cast<float(*)[kStageScalar]>(st);
  const int nbn = (N + 31) / 32, nbc = (E.Cout + 31) / 32;
  const long long plane = (long long)E.Ho * E.Wo;
  const long long cstep = (long long)E.Do * plane;
  const int g = lane & 3;
  for (int blk = warp_e; blk < nbn * nbc; blk += nwarps) {
    const int bn = blk / nbc;
    const int n0 = 32 * bn, c0 = 32 * (blk - bn * nbc);
    const int cg = c0 + 8 * g;
    for (int k = 0; k < 4; ++k) {
      const int pl = 8 * k + (lane >> 2);
      const int n = n0 + pl;
      float y8[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) y8[e] = 0.0f;
      if (n < N && cg < E.Cout) {
        const int cnt = min(8, E.Cout - cg);
        const uint4 raw = *reinterpret_cast<const uint4*>(scr + (long long)n * Cs + cg);
        float v[8];
        unpack8(raw, v);
        const float dn = den[n];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float gm = (e < cnt) ? __ldg(E.gamma + cg + e) : 0.0f;
          y8[e] = norm_silu1(v[e], dn, E.sqrt_c, gm);
        }
        int h, w;
        const bool in_tile = cm_pixel(t, n, h, w);
        if ((E.flags & EPI_SAVE_VALUE) && in_tile && n < t.npix && h < E.Ho && w < E.Wo) {
          const long long o = cm_res_offset(E, t, h, w, cg);
          for (int e = 0; e < cnt; ++e) E.val[o + e * cstep] = bf16_bits(v[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) stage[pl][8 * g + e] = y8[e];
    }
    __syncwarp();
    // lane = pixel n0 + lane: for each channel the warp stores 32 consecutive pixels
    const int n = n0 + lane;
    int h, w;
    const bool in_tile = cm_pixel(t, n, h, w);
    if (n < N && in_tile && n < t.npix && h < E.Ho && w < E.Wo) {
      const long long o = cm_res_offset(E, t, h, w, c0);
      const int cend = min(32, E.Cout - c0);
      for (int c = 0; c < cend; ++c) E.y[o + c * cstep] = bf16_bits(stage[lane][c]);
    }
    __syncwarp();
  }
}

}  // namespace vvc
