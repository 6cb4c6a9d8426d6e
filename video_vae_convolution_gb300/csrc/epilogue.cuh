// Per-pixel epilogue of the convolution: the post-operation contract of the
// cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm + SiLU"
// (section "Operation Contract"), applied to one output pixel's channel row,
// 16 channels at a time.  Every B() rounding point is an explicit
// round-to-nearest-even fp32 -> bf16 conversion, and every fp32 operation is
// an explicitly rounded intrinsic, so nothing is contracted or reassociated.
//
// The row is produced by a loader functor (TMEM accumulators, split-K
// partial sums, or an existing bf16 tensor); loader calls are made the same
// number of times by every thread of a warp, whatever the pixel's validity.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "internal.h"

namespace vvc {

__device__ __forceinline__ uint16_t bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_val(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}
__device__ __forceinline__ float round_bf16(float f) { return bf16_val(bf16_bits(f)); }

struct Pixel {
  int n, d, h, w;
  bool valid;
};

// Element offset of (n, c, d, h, w) in a tensor of the given layout / extent.
__device__ __forceinline__ long long elem_offset(int layout, int C, int D, int H, int W, int n,
                                                 int c, int d, int h, int w) {
  if (layout == LAYOUT_NDHWC)
    return ((((long long)n * D + d) * H + h) * (long long)W + w) * C + c;
  return ((((long long)n * C + c) * D + d) * (long long)H + h) * W + w;
}

// Stores `cnt` (<= 16) consecutive channels starting at c.
__device__ __forceinline__ void store_chunk(uint16_t* base, int layout, int C, int D, int H, int W,
                                            int n, int d, int h, int w, int c, int cnt,
                                            const uint16_t (&v)[16]) {
  if (layout == LAYOUT_NDHWC) {
    uint16_t* p = base + elem_offset(layout, C, D, H, W, n, c, d, h, w);
    if (cnt == 16 && ((reinterpret_cast<uintptr_t>(p) & 15u) == 0)) {
      uint4 a, b;
      a.x = v[0] | (uint32_t(v[1]) << 16);
      a.y = v[2] | (uint32_t(v[3]) << 16);
      a.z = v[4] | (uint32_t(v[5]) << 16);
      a.w = v[6] | (uint32_t(v[7]) << 16);
      b.x = v[8] | (uint32_t(v[9]) << 16);
      b.y = v[10] | (uint32_t(v[11]) << 16);
      b.z = v[12] | (uint32_t(v[13]) << 16);
      b.w = v[14] | (uint32_t(v[15]) << 16);
      reinterpret_cast<uint4*>(p)[0] = a;
      reinterpret_cast<uint4*>(p)[1] = b;
    } else if (cnt == 8 && ((reinterpret_cast<uintptr_t>(p) & 15u) == 0)) {
      uint4 a;
      a.x = v[0] | (uint32_t(v[1]) << 16);
      a.y = v[2] | (uint32_t(v[3]) << 16);
      a.z = v[4] | (uint32_t(v[5]) << 16);
      a.w = v[6] | (uint32_t(v[7]) << 16);
      reinterpret_cast<uint4*>(p)[0] = a;
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < cnt) p[i] = v[i];
    }
  } else {
    const long long plane = (long long)D * H * W;
    uint16_t* p = base + elem_offset(layout, C, D, H, W, n, c, d, h, w);
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if (i < cnt) p[i * plane] = v[i];
  }
}

__device__ __forceinline__ void load_chunk(const uint16_t* base, int layout, int C, int D, int H,
                                           int W, int n, int d, int h, int w, int c, int cnt,
                                           float (&v)[16]) {
  if (layout == LAYOUT_NDHWC) {
    const uint16_t* p = base + elem_offset(layout, C, D, H, W, n, c, d, h, w);
    if (cnt == 16 && ((reinterpret_cast<uintptr_t>(p) & 15u) == 0)) {
      const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
      const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
      const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[2 * i] = __uint_as_float(u[i] << 16);
        v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = (i < cnt) ? bf16_val(p[i]) : 0.0f;
    }
  } else {
    const long long plane = (long long)D * H * W;
    const uint16_t* p = base + elem_offset(layout, C, D, H, W, n, c, d, h, w);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = (i < cnt) ? bf16_val(p[i * plane]) : 0.0f;
  }
}

// acc (fp32) -> value, in place, for channels [c, c + 16); conv bits kept for
// the debug store.  main = B(B(acc) + bias); skip = B(res + rbias);
// value = B(main + skip).
__device__ __forceinline__ void epi_value16(const EpiParams& e, const Pixel& px, int c, int cnt,
                                            float (&v)[16], uint16_t (&convb)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    convb[i] = bf16_bits(v[i]);
    v[i] = bf16_val(convb[i]);
  }
  if (e.flags & EPI_BIAS) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float b = (i < cnt) ? __ldg(e.bias + c + i) : 0.0f;
      v[i] = round_bf16(__fadd_rn(v[i], b));
    }
  }
  if (e.flags & EPI_RESIDUAL) {
    float sk[16];
    if (px.valid) {
      load_chunk(e.residual, e.out_layout, e.Cout, e.Do, e.Ho, e.Wo, px.n, px.d, px.h, px.w, c,
                 cnt, sk);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) sk[i] = 0.0f;
    }
    if (e.flags & EPI_RESIDUAL_BIAS) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float rb = (i < cnt) ? __ldg(e.rbias + c + i) : 0.0f;
        sk[i] = round_bf16(__fadd_rn(sk[i], rb));
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = round_bf16(__fadd_rn(v[i], sk[i]));
  }
}

// value -> activated: normalized = B(value / den); scaled = B(normalized * sqrt(C));
// affine = B(scaled * gamma); activated = B(affine / (1 + exp(-affine))).
__device__ __forceinline__ float norm_silu1(float v, float den, float sqrt_c, float g) {
  const float nrm = round_bf16(__fdiv_rn(v, den));
  const float sc = round_bf16(__fmul_rn(nrm, sqrt_c));
  const float af = round_bf16(__fmul_rn(sc, g));
  const float ex = expf(-af);
  return round_bf16(__fdiv_rn(af, __fadd_rn(1.0f, ex)));
}

// den = max(sqrt(sum of squares), 1e-12)
__device__ __forceinline__ float norm_den(float ss) {
  const float den = __fsqrt_rn(ss);
  return (den > 1e-12f) ? den : 1e-12f;
}

__device__ __forceinline__ void epi_norm_silu16(const EpiParams& e, int c, int cnt, float den,
                                                float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g = (i < cnt) ? __ldg(e.gamma + c + i) : 0.0f;
    v[i] = norm_silu1(v[i], den, e.sqrt_c, g);
  }
}

// Halo positions along one axis of a haloed y that take output coordinate i
// besides i itself (extent L; at most one halo pixel before and after), as bits:
// 1 = position -1, 4 = position L, with 2 / 8 marking a zero fill of that position.
// Reflection (mode 2): -1 holds 1, L holds L - 2; zeros (mode 1): -1 beside 0, L
// beside L - 1.
__device__ __forceinline__ int halo_bits(int i, int L, int before, int after, int mode) {
  int b = 0;
  if (mode == 2) {
    if (before && i == 1) b |= 1;
    if (after && i == L - 2) b |= 4;
  } else if (mode == 1) {
    if (before && i == 0) b |= 3;
    if (after && i == L - 1) b |= 12;
  }
  return b;
}

// Element offset in a haloed NDHWC y of channel c of output pixel (n, d, h, w),
// h and w in output coordinates (-1 .. L for the halo).
__device__ __forceinline__ long long halo_offset(const EpiParams& e, int n, int d, int h, int w,
                                                 int c) {
  return ((((long long)n * e.Dy + d + e.d0) * e.Hy + h + e.h0) * (long long)e.Wy + w + e.w0) *
             e.Cout + c;
}

// Calls put(offset, zero) for every halo position of a haloed y that output pixel
// (n, d, h, w) fills besides its own (reflected copies and zero neighbours), with
// offset the element offset of channel c there.
template <class Put>
__device__ __forceinline__ void halo_extras(const EpiParams& e, int n, int d, int h, int w, int c,
                                            Put&& put) {
  const int bh = halo_bits(h, e.Ho, e.h0, e.Hy - e.Ho - e.h0, e.h_mode);
  const int bw = halo_bits(w, e.Wo, e.w0, e.Wy - e.Wo - e.w0, e.w_mode);
  if ((bh | bw) == 0) return;
  // the halo columns of one row (hh), zero when the row or the column is a zero fill
  auto cols = [&](int hh, bool zr) {
    if (bw & 1) put(halo_offset(e, n, d, hh, -1, c), zr || (bw & 2));
    if (bw & 4) put(halo_offset(e, n, d, hh, e.Wo, c), zr || (bw & 8));
  };
  cols(h, false);
  if (bh & 1) {
    put(halo_offset(e, n, d, -1, w, c), (bh & 2) != 0);
    cols(-1, (bh & 2) != 0);
  }
  if (bh & 4) {
    put(halo_offset(e, n, d, e.Ho, w, c), (bh & 8) != 0);
    cols(e.Ho, (bh & 8) != 0);
  }
}

// Writes y (and value_out / conv_out) for one chunk of one pixel; adds the
// zero bottom row / right column of OUT_PAD_BR next to border pixels, and the
// halo copies of a haloed y.
__device__ __forceinline__ void epi_store16(const EpiParams& e, const Pixel& px, int c, int cnt,
                                            const float (&y)[16], const uint16_t (&yb_in)[16],
                                            bool use_bits) {
  uint16_t yb[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) yb[i] = use_bits ? yb_in[i] : bf16_bits(y[i]);
  const bool pad = (e.flags & EPI_OUT_PAD_BR) != 0;
  const int Hy = e.Ho + (pad ? 1 : 0), Wy = e.Wo + (pad ? 1 : 0);
  uint16_t* yp = static_cast<uint16_t*>(e.y);
  if (e.halo) {
    // NDHWC: the pixel's own position, then its reflected copies / zero neighbours
    auto put = [&](long long off, bool zero) {
      uint16_t* q = yp + off;
      if ((cnt == 8 || cnt == 16) && ((reinterpret_cast<uintptr_t>(q) & 15u) == 0)) {
        // 16-byte stores of 8 channels
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          if (k * 8 >= cnt) break;
          uint4 a = make_uint4(0u, 0u, 0u, 0u);
          if (!zero) {
            a.x = yb[8 * k] | (uint32_t(yb[8 * k + 1]) << 16);
            a.y = yb[8 * k + 2] | (uint32_t(yb[8 * k + 3]) << 16);
            a.z = yb[8 * k + 4] | (uint32_t(yb[8 * k + 5]) << 16);
            a.w = yb[8 * k + 6] | (uint32_t(yb[8 * k + 7]) << 16);
          }
          reinterpret_cast<uint4*>(q)[k] = a;
        }
        return;
      }
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < cnt) q[i] = zero ? uint16_t(0) : yb[i];
    };
    put(halo_offset(e, px.n, px.d, px.h, px.w, c), false);
    halo_extras(e, px.n, px.d, px.h, px.w, c, put);
    return;
  }
  store_chunk(yp, e.out_layout, e.Cout, e.Do, Hy, Wy, px.n, px.d, px.h, px.w, c, cnt, yb);
  if (pad) {
    uint16_t z[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = 0;
    const bool last_w = (px.w == e.Wo - 1), last_h = (px.h == e.Ho - 1);
    if (last_w) store_chunk(yp, e.out_layout, e.Cout, e.Do, Hy, Wy, px.n, px.d, px.h, e.Wo, c, cnt, z);
    if (last_h) store_chunk(yp, e.out_layout, e.Cout, e.Do, Hy, Wy, px.n, px.d, e.Ho, px.w, c, cnt, z);
    if (last_w && last_h)
      store_chunk(yp, e.out_layout, e.Cout, e.Do, Hy, Wy, px.n, px.d, e.Ho, e.Wo, c, cnt, z);
  }
}

// Full epilogue of one pixel over channels [cb, ce).  With L2NORM_SILU the
// range must be the whole row [0, Cout).  `load(c_rel, v)` returns 16 fp32
// values for channels cb + c_rel ...; it is called uniformly across the warp.
template <class Loader>
__device__ __forceinline__ void epilogue_pixel(const EpiParams& e, const Pixel& px, int cb, int ce,
                                               Loader&& load) {
  const bool norm = (e.flags & EPI_L2NORM_SILU) != 0;
  float den = 1.0f;
  if (norm) {
    // den = max(sqrt(sum over the row of value^2), 1e-12), summed in channel order
    float ss = 0.0f;
    for (int c = cb; c < ce; c += 16) {
      const int cnt = min(16, ce - c);
      float v[16];
      uint16_t cv[16];
      load(c - cb, v);
      epi_value16(e, px, c, cnt, v, cv);
#pragma unroll
      for (int i = 0; i < 16; ++i)
        if (i < cnt) ss = __fadd_rn(ss, __fmul_rn(v[i], v[i]));
    }
    den = norm_den(ss);
  }
  for (int c = cb; c < ce; c += 16) {
    const int cnt = min(16, ce - c);
    float v[16];
    uint16_t cv[16];
    load(c - cb, v);
    epi_value16(e, px, c, cnt, v, cv);
    if (!px.valid) continue;
    if (e.flags & EPI_DEBUG_STORE_CONV)
      store_chunk(e.conv_out, LAYOUT_NDHWC, e.Cout, e.Do, e.Ho, e.Wo, px.n, px.d, px.h, px.w, c,
                  cnt, cv);
    if (e.flags & EPI_SAVE_VALUE) {
      uint16_t vb[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) vb[i] = bf16_bits(v[i]);
      store_chunk(e.value_out, e.out_layout, e.Cout, e.Do, e.Ho, e.Wo, px.n, px.d, px.h, px.w, c,
                  cnt, vb);
    }
    if (norm) epi_norm_silu16(e, c, cnt, den, v);
    epi_store16(e, px, c, cnt, v, cv, false);
  }
}

}  // namespace vvc
