// Memory-bound companions of the tensor-core convolution:
//  - weight pack OITRS -> OTRSI with Cin padded to 64 (cuDNN frontend doc
//    "Fused Conv3D + Bias + Residual + RMSNorm + SiLU", "Weight Packing");
//  - input staging into channels-last (NCDHW -> NDHWC transpose, or channel
//    padding to a multiple of 8 so TMA strides stay 16-byte multiples);
//  - the deterministic split-K reduction + epilogue (ROCm/FlyDSL issue
//    "[Feature]: conv3d_implicit — ...", maintainer comment: the split-K path
//    materialises an NDHWC-flat (npq, k) buffer then reduces);
//  - the standalone post-operations (cuDNN doc, "Standalone Normalization and
//    Padding Variant", contiguous output).
#include <cuda_runtime.h>

#include <algorithm>

#include "epilogue.cuh"
#include "internal.h"
#include "pad_cache.h"

namespace vvc {

// ---- weight pack -------------------------------------------------------------------
__global__ void pack_weight_kernel(const uint16_t* __restrict__ w, uint16_t* __restrict__ out,
                                   int Co, int Ci, int taps, int cp, long long total) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ci = static_cast<int>(i % cp);
    const long long rest = i / cp;
    const int tap = static_cast<int>(rest % taps);
    const long long co = rest / taps;
    out[i] = (ci < Ci) ? w[(co * Ci + ci) * taps + tap] : uint16_t(0);
  }
}

cudaError_t launch_pack_weight(const void* w, void* out, int Co, int Ci, int taps,
                               cudaStream_t s) {
  const int cp = (Ci + 63) / 64 * 64;
  const long long total = (long long)Co * taps * cp;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  pack_weight_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(
      static_cast<const uint16_t*>(w), static_cast<uint16_t*>(out), Co, Ci, taps, cp, total);
  return cudaGetLastError();
}

// One-byte (e4m3) weights: OITRS -> OTRSI with Ci zero-padded to a multiple of 128;
// a thread writes one 16-byte group of 16 input channels of one (co, tap).
__global__ void pack_weight_u8_kernel(const uint8_t* __restrict__ w, uint8_t* __restrict__ out,
                                      int Ci, int taps, int groups, long long total) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int g = static_cast<int>(i % groups);
    const long long rest = i / groups;  // co * taps + tap
    const int tap = static_cast<int>(rest % taps);
    const long long co = rest / taps;
    uint32_t v[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int ci = g * 16 + k;
      const uint32_t b = (ci < Ci) ? w[(co * Ci + ci) * taps + tap] : 0u;
      v[k >> 2] |= b << (8 * (k & 3));
    }
    *reinterpret_cast<uint4*>(out + i * 16) = make_uint4(v[0], v[1], v[2], v[3]);
  }
}

cudaError_t launch_pack_weight_u8(const void* w, void* out, int Co, int Ci, int taps,
                                  cudaStream_t s) {
  const int groups = (Ci + 127) / 128 * 8;  // 16-byte groups per (co, tap) row
  const long long total = (long long)Co * taps * groups;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152 * 32) blocks = 152 * 32;
  pack_weight_u8_kernel<<<static_cast<int>(blocks), threads, 0, s>>>(
      static_cast<const uint8_t*>(w), static_cast<uint8_t*>(out), Ci, taps, groups, total);
  return cudaGetLastError();
}

// ---- spatial im2col staging for narrow inputs ------------------------------------------
// For a layer with few input channels (Cin * KR * KS <= 64) the spatial taps are
// gathered once: out[n][d][ho][wo][(r * KS + s) * C + c] = x[n, c, d, ho*sh + r - ph,
// wo*sw + s - pw] (zero or reflect padding; channels past KR*KS*C are zero), so the
// convolution that follows is (KT, 1, 1) over Ck channels, and its weights are
// repacked to match: wr[co][t][(r * KS + s) * C + c] = wp[co][(t*KR + r)*KS + s][c].
// The last `wblocks` blocks of the grid do the weight repack.
struct Im2colArgs {
  const uint16_t* x;
  int layout;                 // LAYOUT_NCDHW / LAYOUT_NDHWC
  int N, C, D, H, W, Ho, Wo;
  int KT, KR, KS, sh, sw, ph, pw, reflect_h, reflect_w;
  int Ck;                     // staged channels (multiple of 8)
  uint16_t* out;
  const uint16_t* wp;         // packed weights [Cout][KT*KR*KS][cp]
  int Cout, cp;               // cp = round_up(C, 64)
  int cp2;                    // round_up(Ck, 64): channel pitch of the repacked weights
  uint16_t* wr;               // [Cout][KT][cp2]
  long long units;            // N * D * Ho * Wo * (Ck / 8)
  int iblocks;                // blocks doing the gather
};

__device__ __forceinline__ int pad_index(int i, int L, bool reflect) {
  if (reflect) {
    if (i < 0) i = -i;
    if (i >= L) i = 2 * (L - 1) - i;
  }
  return i;  // out of [0, L) means zero padding
}

// The weight repack, block b of nb.
__device__ __forceinline__ void im2col_repack_weights(const Im2colArgs& a, int b, int nb) {
  const long long total = (long long)a.Cout * a.KT * a.cp2;
  const int krs = a.KR * a.KS * a.C;
  for (long long i = (long long)b * blockDim.x + threadIdx.x; i < total;
       i += (long long)nb * blockDim.x) {
    const int kk = static_cast<int>(i % a.cp2);
    const long long rest = i / a.cp2;
    const int t = static_cast<int>(rest % a.KT);
    const long long co = rest / a.KT;
    uint16_t v = 0;
    if (kk < krs) {
      const int rs = kk / a.C, c = kk - rs * a.C;
      const int tap = t * a.KR * a.KS + rs;
      v = a.wp[(co * a.KT * a.KR * a.KS + tap) * a.cp + c];
    }
    a.wr[i] = v;
  }
}

// Grid: x = 256-pixel pieces of an output row, y = output row ho, z = n * D + d;
// blockIdx.x past the row pieces (x >= xblocks) repacks the weights.
__global__ void __launch_bounds__(256) im2col_hw_kernel(const Im2colArgs a) {
  const int xblocks = (a.Wo + 255) / 256;
  if (static_cast<int>(blockIdx.x) >= xblocks) {
    if (blockIdx.y != 0 || blockIdx.z != 0) return;
    im2col_repack_weights(a, blockIdx.x - xblocks, gridDim.x - xblocks);
    return;
  }
  const int wo = blockIdx.x * 256 + threadIdx.x;
  if (wo >= a.Wo) return;
  const int ho = blockIdx.y;
  const int nd = blockIdx.z;
  const int n = nd / a.D, d = nd - n * a.D;
  const long long plane = (long long)a.H * a.W;
  const long long cstride = (a.layout == LAYOUT_NDHWC) ? 1 : (long long)a.D * plane;
  const long long base = (a.layout == LAYOUT_NDHWC)
                             ? ((long long)n * a.D + d) * plane * a.C
                             : ((long long)n * a.C * a.D + d) * plane;
  const int pix_stride = (a.layout == LAYOUT_NDHWC) ? a.C : 1;
  uint4* dst = reinterpret_cast<uint4*>(a.out) +
               ((((long long)nd * a.Ho + ho) * a.Wo + wo) * (a.Ck / 8));
  // values are appended 16 bits at a time to (lo, hi); every 8 form one 16-byte store
  unsigned long long lo = 0, hi = 0;
  int ne = 0, g = 0;
  for (int r = 0; r < a.KR; ++r) {
    const int h = pad_index(ho * a.sh + r - a.ph, a.H, a.reflect_h);
    for (int s = 0; s < a.KS; ++s) {
      const int w = pad_index(wo * a.sw + s - a.pw, a.W, a.reflect_w);
      const bool in = h >= 0 && h < a.H && w >= 0 && w < a.W;
      const long long pos = base + ((long long)h * a.W + w) * pix_stride;
      for (int c = 0; c < a.C; ++c) {
        const unsigned long long val = in ? __ldg(a.x + pos + c * cstride) : 0u;
        if (ne < 4)
          lo |= val << (16 * ne);
        else
          hi |= val << (16 * (ne - 4));
        if (++ne == 8) {
          dst[g++] = make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                                static_cast<uint32_t>(hi), static_cast<uint32_t>(hi >> 32));
          lo = hi = 0;
          ne = 0;
        }
      }
    }
  }
  // the rest of the Ck channels are zero
  for (; g < a.Ck / 8; ++g) {
    dst[g] = make_uint4(static_cast<uint32_t>(lo), static_cast<uint32_t>(lo >> 32),
                        static_cast<uint32_t>(hi), static_cast<uint32_t>(hi >> 32));
    lo = hi = 0;
  }
}

// The same gather for 3 x 3 spatial taps and a fixed channel count: every tap's
// loads are issued before the values are packed (the loop above waits for each
// load in turn).
template <int C>
// Grid: x = 256-pixel pieces of an output row, y = output row ho, z = n * D + d, plus one
// more z slice whose blocks (x = 0, y < wblocks) repack the weights alongside the gather.
__global__ void __launch_bounds__(256) im2col_3x3_kernel(const Im2colArgs a, int wblocks) {
  const int xblocks = (a.Wo + 255) / 256;
  if (static_cast<int>(blockIdx.z) == a.N * a.D) {
    if (blockIdx.x == 0 && static_cast<int>(blockIdx.y) < wblocks)
      im2col_repack_weights(a, blockIdx.y, wblocks);
    return;
  }
  if (static_cast<int>(blockIdx.x) >= xblocks) return;
  const int wo = blockIdx.x * 256 + threadIdx.x;
  if (wo >= a.Wo) return;
  const int ho = blockIdx.y;
  const int nd = blockIdx.z;
  const int n = nd / a.D, d = nd - n * a.D;
  const long long plane = (long long)a.H * a.W;
  const long long cstride = (a.layout == LAYOUT_NDHWC) ? 1 : (long long)a.D * plane;
  const long long base = (a.layout == LAYOUT_NDHWC)
                             ? ((long long)n * a.D + d) * plane * C
                             : ((long long)n * C * a.D + d) * plane;
  const int pix_stride = (a.layout == LAYOUT_NDHWC) ? C : 1;
  constexpr int kVals = 9 * C;
  constexpr int kGroups = (kVals + 7) / 8;
  uint16_t v[kGroups * 8];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int h = pad_index(ho * a.sh + r - a.ph, a.H, a.reflect_h);
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const int w = pad_index(wo * a.sw + s - a.pw, a.W, a.reflect_w);
      const bool in = h >= 0 && h < a.H && w >= 0 && w < a.W;
      const long long pos = base + ((long long)(in ? h : 0) * a.W + (in ? w : 0)) * pix_stride;
#pragma unroll
      for (int c = 0; c < C; ++c)
        v[(r * 3 + s) * C + c] = in ? __ldg(a.x + pos + c * cstride) : uint16_t(0);
    }
  }
#pragma unroll
  for (int e = kVals; e < kGroups * 8; ++e) v[e] = 0;
  uint4* dst = reinterpret_cast<uint4*>(a.out) +
               ((((long long)nd * a.Ho + ho) * a.Wo + wo) * (a.Ck / 8));
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    uint4 q;
    q.x = v[8 * g] | (uint32_t(v[8 * g + 1]) << 16);
    q.y = v[8 * g + 2] | (uint32_t(v[8 * g + 3]) << 16);
    q.z = v[8 * g + 4] | (uint32_t(v[8 * g + 5]) << 16);
    q.w = v[8 * g + 6] | (uint32_t(v[8 * g + 7]) << 16);
    dst[g] = q;
  }
  for (int g = kGroups; g < a.Ck / 8; ++g) dst[g] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_im2col_hw(const void* x, int layout, int N, int C, int D, int H, int W, int Ho,
                             int Wo, int KT, int KR, int KS, int sh, int sw, int ph, int pw,
                             int reflect_h, int reflect_w, int Ck, void* out, const void* wp,
                             int Cout, void* wr, cudaStream_t s) {
  Im2colArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.layout = layout;
  a.N = N; a.C = C; a.D = D; a.H = H; a.W = W; a.Ho = Ho; a.Wo = Wo;
  a.KT = KT; a.KR = KR; a.KS = KS; a.sh = sh; a.sw = sw; a.ph = ph; a.pw = pw;
  a.reflect_h = reflect_h; a.reflect_w = reflect_w;
  a.Ck = Ck;
  a.out = static_cast<uint16_t*>(out);
  a.wp = static_cast<const uint16_t*>(wp);
  a.Cout = Cout;
  a.cp = (C + 63) / 64 * 64;
  a.cp2 = (Ck + 63) / 64 * 64;
  a.wr = static_cast<uint16_t*>(wr);
  a.units = (long long)N * D * Ho * Wo * (Ck / 8);
  const int xblocks = (Wo + 255) / 256;
  a.iblocks = xblocks;
  // blocks that repack the weights beside the generic gather (the extra blocks of its
  // grid), and in a launch of their own after the 3 x 3 gather: enough there to finish
  // in about a microsecond (8 blocks took 13 us for the 128 x 3 x 64 repacked weights
  // of the RGB input convolution)
  const int wblocks = 8;
  const long long wtotal = (long long)Cout * KT * a.cp2;
  const int wblocks_own =
      static_cast<int>(std::min<long long>(152, std::max<long long>(1, (wtotal + 2047) / 2048)));
  if (KR == 3 && KS == 3 && C >= 1 && C <= 7 && (long long)N * D < 65535) {
    // gather through the unrolled kernel, the weight repack in the same launch (blocks of
    // an extra z slice, up to Ho of them)
    const int wb = std::min(wblocks_own, Ho);
    const dim3 g(xblocks, Ho, N * D + 1);
    switch (C) {
      case 1: im2col_3x3_kernel<1><<<g, 256, 0, s>>>(a, wb); break;
      case 2: im2col_3x3_kernel<2><<<g, 256, 0, s>>>(a, wb); break;
      case 3: im2col_3x3_kernel<3><<<g, 256, 0, s>>>(a, wb); break;
      case 4: im2col_3x3_kernel<4><<<g, 256, 0, s>>>(a, wb); break;
      case 5: im2col_3x3_kernel<5><<<g, 256, 0, s>>>(a, wb); break;
      case 6: im2col_3x3_kernel<6><<<g, 256, 0, s>>>(a, wb); break;
      default: im2col_3x3_kernel<7><<<g, 256, 0, s>>>(a, wb); break;
    }
    return cudaGetLastError();
  }
  im2col_hw_kernel<<<dim3(xblocks + wblocks, Ho, N * D), 256, 0, s>>>(a);
  return cudaGetLastError();
}

// ---- input staging --------------------------------------------------------------------
// NCDHW [N][C][S] (S = D*H*W) -> NDHWC [N][S][Cp], channels Cin..Cp-1 zero.
// S % 8 == 0: a thread moves an 8-channel x 8-position block in registers: eight 16-byte
// loads (8 positions of one channel each), a transpose of the 8 x 8 bf16 block by byte
// permutes, eight 16-byte stores (8 channels of one position each).  A warp covers 4
// channel groups x 8 position groups, so each load instruction reads 128 contiguous
// bytes of 4 channel rows and each store writes 64 contiguous bytes of 8 positions.
// Grid: x = 512-position pieces, y = 32-channel pieces of Cp, z = batch.
__global__ void __launch_bounds__(256) ncdhw_to_ndhwc_r8_kernel(const uint16_t* __restrict__ x,
                                                                uint16_t* __restrict__ out,
                                                                int C, int Cp, long long S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = blockIdx.y * 4 + (lane & 3);                        // channel group
  const long long q = (long long)blockIdx.x * 64 + warp * 8 + (lane >> 2);  // position group
  if (8 * g >= Cp || 8 * q >= S) return;
  const uint16_t* xn = x + (long long)blockIdx.z * C * S;
  uint16_t* on = out + (long long)blockIdx.z * Cp * S;
  uint4 v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int c = 8 * g + k;
    v[k] = (c < C) ? __ldg(reinterpret_cast<const uint4*>(xn + (long long)c * S + 8 * q))
                   : make_uint4(0u, 0u, 0u, 0u);
  }
  auto word = [](const uint4& a, int i) { return i == 0 ? a.x : (i == 1 ? a.y : (i == 2 ? a.z : a.w)); };
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    // position 8q + j: channel 8g + k is element j of v[k]
    const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
    uint4 o;
    o.x = __byte_perm(word(v[0], j >> 1), word(v[1], j >> 1), sel);
    o.y = __byte_perm(word(v[2], j >> 1), word(v[3], j >> 1), sel);
    o.z = __byte_perm(word(v[4], j >> 1), word(v[5], j >> 1), sel);
    o.w = __byte_perm(word(v[6], j >> 1), word(v[7], j >> 1), sel);
    *reinterpret_cast<uint4*>(on + (8 * q + j) * Cp + 8 * g) = o;
  }
}

// Any S: a block moves 32 channels x 256 positions through shared memory; each
// channel row is read as 512 contiguous bytes (2-byte loads), and each position's
// 32 channels are written as four 16-byte stores by four neighbouring lanes.
__global__ void __launch_bounds__(256)
    ncdhw_to_ndhwc_scalar_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out, int C,
                                 int Cp, long long S) {
  __shared__ uint16_t tile[32][256 + 2];  // odd word pitch: conflict-free column reads
  const int n = blockIdx.z;
  const long long s0 = (long long)blockIdx.x * 256;
  const int c0 = blockIdx.y * 32;
  const uint16_t* xn = x + (long long)n * C * S;
  uint16_t* on = out + (long long)n * Cp * S;
  const int tid = threadIdx.x;
  const long long s = s0 + tid;
  for (int k = 0; k < 32; ++k) {
    const int c = c0 + k;
    tile[k][tid] = (c < C && s < S) ? xn[(long long)c * S + s] : uint16_t(0);
  }
  __syncthreads();
  const int nch = min(32, Cp - c0);     // channels of this block present in the output
  const int groups = (nch + 7) / 8;     // 16-byte groups per position (Cp % 8 == 0)
  for (int u = tid; u < 256 * 4; u += 256) {
    const int pl = u >> 2, g = u & 3;
    const long long sp = s0 + pl;
    if (g >= groups || sp >= S) continue;
    uint16_t v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = tile[8 * g + e][pl];
    uint4 q;
    q.x = v[0] | (uint32_t(v[1]) << 16);
    q.y = v[2] | (uint32_t(v[3]) << 16);
    q.z = v[4] | (uint32_t(v[5]) << 16);
    q.w = v[6] | (uint32_t(v[7]) << 16);
    *reinterpret_cast<uint4*>(on + sp * Cp + c0 + 8 * g) = q;
  }
}


// NDHWC [P][C] -> [P][Cp] with zero channels Cin..Cp-1.
__global__ void pad_channels_kernel(const uint16_t* __restrict__ x, uint16_t* __restrict__ out,
                                    int C, int Cp, long long P) {
  const long long total = P * Cp;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int c = static_cast<int>(i % Cp);
    const long long p = i / Cp;
    out[i] = (c < C) ? x[p * C + c] : uint16_t(0);
  }
}

cudaError_t launch_stage_input(const void* x, int layout, int N, int C, int Cp, long long S,
                               void* out, cudaStream_t s) {
  if (layout == LAYOUT_NCDHW) {
    const bool vec = (S % 8) == 0 && (reinterpret_cast<uintptr_t>(x) % 16) == 0;
    if (vec) {
      dim3 grid(static_cast<unsigned>((S / 8 + 63) / 64), static_cast<unsigned>((Cp + 31) / 32),
                static_cast<unsigned>(N));
      ncdhw_to_ndhwc_r8_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x),
                                                    static_cast<uint16_t*>(out), C, Cp, S);
    } else {
      dim3 grid(static_cast<unsigned>((S + 255) / 256), static_cast<unsigned>((Cp + 31) / 32),
                static_cast<unsigned>(N));
      ncdhw_to_ndhwc_scalar_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x),
                                                        static_cast<uint16_t*>(out), C, Cp, S);
    }
  } else {
    const long long total = (long long)N * S * Cp;
    long long blocks = (total + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    pad_channels_kernel<<<static_cast<int>(blocks), 256, 0, s>>>(
        static_cast<const uint16_t*>(x), static_cast<uint16_t*>(out), C, Cp, (long long)N * S);
  }
  return cudaGetLastError();
}

// ---- split-K reduction + epilogue ----------------------------------------------------------
// partial: [splits][M][Cout] fp32, NDHWC-flat pixels.  One thread per pixel, the
// splits summed in index order (deterministic).
__global__ void splitk_epilogue_kernel(const float* __restrict__ partial, int splits,
                                       long long M, EpiParams e) {
  const long long pix = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  Pixel px;
  px.valid = pix < M;
  const long long pp = px.valid ? pix : 0;
  px.w = static_cast<int>(pp % e.Wo);
  long long rest = pp / e.Wo;
  px.h = static_cast<int>(rest % e.Ho);
  rest /= e.Ho;
  px.d = static_cast<int>(rest % e.Do);
  px.n = static_cast<int>(rest / e.Do);
  const bool vec = (e.Cout % 4) == 0;
  auto load = [&](int c_rel, float(&v)[16]) {
    const int c = c_rel;
    const int cnt = min(16, e.Cout - c);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    if (!px.valid) return;
    for (int s = 0; s < splits; ++s) {
      const float* src = partial + ((long long)s * M + pp) * e.Cout + c;
      if (vec && cnt == 16) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(src) + k);
          v[4 * k] += q.x;
          v[4 * k + 1] += q.y;
          v[4 * k + 2] += q.z;
          v[4 * k + 3] += q.w;
        }
      } else {
        for (int i = 0; i < cnt; ++i) v[i] += __ldg(src + i);
      }
    }
  };
  epilogue_pixel(e, px, 0, e.Cout, load);
}

// Same reduction when the epilogue is per element (no L2 norm): one thread per
// (pixel, 16-channel chunk), so small layers still spread over every SM; adjacent
// threads read and write adjacent 64-byte chunks of a pixel row.
// One thread per (pixel, `width` channels): width 8 when Cout % 8 == 0 (16-byte
// output stores, twice the threads of width 16), else 16.  The partial sums are added
// in split order from 0 (deterministic); the loads of four splits are issued before
// their additions so that they overlap.
__global__ void splitk_epilogue_chunk_kernel(const float* __restrict__ partial, int splits,
                                             long long M, EpiParams e, int width) {
  const int chunks = (e.Cout + width - 1) / width;
  const long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  Pixel px;
  px.valid = u < M * chunks;
  const long long uu = px.valid ? u : 0;
  const long long pp = uu / chunks;
  const int c0 = static_cast<int>(uu - pp * chunks) * width;
  px.w = static_cast<int>(pp % e.Wo);
  long long rest = pp / e.Wo;
  px.h = static_cast<int>(rest % e.Ho);
  rest /= e.Ho;
  px.d = static_cast<int>(rest % e.Do);
  px.n = static_cast<int>(rest / e.Do);
  const int cnt = min(width, e.Cout - c0);
  const bool vec = (e.Cout % 4) == 0 && cnt == 16;
  const bool vec8 = (e.Cout % 8) == 0 && width == 8;
  auto load = [&](int c_rel, float(&v)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.0f;
    if (!px.valid) return;
    if (vec8) {
      const float* base = partial + pp * e.Cout + c0 + c_rel;
      const long long sstride = M * e.Cout;
      int s = 0;
      for (; s + 4 <= splits; s += 4) {
        float4 a[4][2];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4* q = reinterpret_cast<const float4*>(base + (s + k) * sstride);
          a[k][0] = __ldg(q);
          a[k][1] = __ldg(q + 1);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[0] += a[k][0].x; v[1] += a[k][0].y; v[2] += a[k][0].z; v[3] += a[k][0].w;
          v[4] += a[k][1].x; v[5] += a[k][1].y; v[6] += a[k][1].z; v[7] += a[k][1].w;
        }
      }
      for (; s < splits; ++s) {
        const float4* q = reinterpret_cast<const float4*>(base + s * sstride);
        const float4 lo = __ldg(q), hi = __ldg(q + 1);
        v[0] += lo.x; v[1] += lo.y; v[2] += lo.z; v[3] += lo.w;
        v[4] += hi.x; v[5] += hi.y; v[6] += hi.z; v[7] += hi.w;
      }
      return;
    }
    for (int s = 0; s < splits; ++s) {
      const float* src = partial + ((long long)s * M + pp) * e.Cout + c0 + c_rel;
      if (vec) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 q = __ldg(reinterpret_cast<const float4*>(src) + k);
          v[4 * k] += q.x;
          v[4 * k + 1] += q.y;
          v[4 * k + 2] += q.z;
          v[4 * k + 3] += q.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (i < cnt) v[i] += __ldg(src + i);
      }
    }
  };
  epilogue_pixel(e, px, c0, c0 + cnt, load);
}

cudaError_t launch_splitk_epilogue(const float* partial, int splits, long long M,
                                   const EpiParams& e, cudaStream_t s) {
  const int threads = 128;
  if (!(e.flags & EPI_L2NORM_SILU)) {
    const int width = (e.Cout % 8 == 0) ? 8 : 16;
    const long long units = M * ((e.Cout + width - 1) / width);
    const long long blocks = (units + threads - 1) / threads;
    splitk_epilogue_chunk_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
        partial, splits, M, e, width);
    return cudaGetLastError();
  }
  const long long blocks = (M + threads - 1) / threads;
  splitk_epilogue_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(partial, splits, M, e);
  return cudaGetLastError();
}

// ---- standalone post-operations ------------------------------------------------------------
// x: [rows][C] bf16.  One thread per row; the epilogue addressing sees the rows as
// an NDHWC tensor of extent (1, 1, 1, rows, C).
__global__ void l2norm_silu_kernel(const uint16_t* __restrict__ x, long long rows, EpiParams e) {
  const long long row = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  Pixel px;
  px.valid = row < rows;
  px.n = 0;
  px.d = 0;
  px.h = 0;
  px.w = static_cast<int>(px.valid ? row : 0);
  const int C = e.Cout;
  auto load = [&](int c_rel, float(&v)[16]) {
    const int cnt = min(16, C - c_rel);
    if (!px.valid) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.0f;
      return;
    }
    load_chunk(x, LAYOUT_NDHWC, C, 1, 1, e.Wo, 0, 0, 0, px.w, c_rel, cnt, v);
  };
  epilogue_pixel(e, px, 0, C, load);
}

cudaError_t launch_norm_rows(const void* x, long long rows, const EpiParams& e, int T, int H,
                             int W, int padded, cudaStream_t s);
size_t norm_rows_smem(int C, int R);

cudaError_t launch_l2norm_silu(const void* x, long long rows, const EpiParams& e,
                               cudaStream_t s) {
  if (e.Cout % 8 == 0 && norm_rows_smem(e.Cout, 1) != 0)  // 16-byte rows: staged kernel
    return launch_norm_rows(x, rows, e, 1, 1, 1, 0, s);
  const int threads = 128;
  const long long blocks = (rows + threads - 1) / threads;
  l2norm_silu_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(
      static_cast<const uint16_t*>(x), rows, e);
  return cudaGetLastError();
}

// ---- padded output + two-frame cache (cuDNN frontend doc "Fused Conv3D + Bias +
//      Residual + RMSNorm + SiLU", "Normalization and Padding Variant" and
//      "Standalone Normalization and Padding Variant") ---------------------------------

// Standalone post-operations, C % 8 == 0, rows staged through shared memory.  A
// block takes R consecutive rows (pixels) of x:
//   1. every element's value = B(B(x + bias) + B(residual + residual_bias)) (steps
//      as the flags ask) is computed from 16-byte loads, coalesced across the block,
//      and kept as bf16 in shared memory (value_out written here);
//   2. one thread per row sums value^2 in channel order: den = max(sqrt(.), 1e-12);
//   3. every element's activation B(B(B(B(value / den) * sqrt(C)) * gamma) / (1 +
//      exp(-.))) goes out in 16-byte stores, to row r of y or (padded) to the
//      interior position (n, t + 2, h + 1, w + 1) of [N, T + 2, H + 2, W + 2, C].
// The rounding steps and the order of the sum are those of epilogue_pixel.
constexpr int kNormRows = 32;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = uint32_t(bf16_bits(f[2 * i])) | (uint32_t(bf16_bits(f[2 * i + 1])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(256) l2norm_silu_rows_kernel(const uint16_t* __restrict__ x,
                                                               long long rows, EpiParams e,
                                                               int T, int H, int W, int padded,
                                                               int R) {
  extern __shared__ uint4 norm_smem[];
  const int C = e.Cout;
  const int G = C >> 3;          // 16-byte groups per row
  const int pitch = G + 1;       // staged row pitch in 16-byte words
  uint4* stage = norm_smem;
  float* den = reinterpret_cast<float*>(norm_smem + (size_t)R * pitch);
  long long* dst_row = reinterpret_cast<long long*>(den + R + (R & 1));
  const long long r0 = (long long)blockIdx.x * R;
  const int nr = static_cast<int>(rows - r0 < R ? rows - r0 : R);
  const bool bias = (e.flags & EPI_BIAS) != 0, res = (e.flags & EPI_RESIDUAL) != 0;
  const bool rbias = (e.flags & EPI_RESIDUAL_BIAS) != 0, save = (e.flags & EPI_SAVE_VALUE) != 0;
  for (int u = threadIdx.x; u < nr * G; u += blockDim.x) {
    const int r = u / G, g = u - r * G;
    const long long off = (r0 + r) * C + 8 * g;
    float v[8];
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + off), v);
    if (bias) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = round_bf16(__fadd_rn(v[i], __ldg(e.bias + 8 * g + i)));
    }
    if (res) {
      float sk[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(e.residual + off), sk);
      if (rbias) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          sk[i] = round_bf16(__fadd_rn(sk[i], __ldg(e.rbias + 8 * g + i)));
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = round_bf16(__fadd_rn(v[i], sk[i]));
    }
    const uint4 vb = f32_to_bf16x8(v);
    stage[r * pitch + g] = vb;
    if (save) *reinterpret_cast<uint4*>(e.value_out + off) = vb;
  }
  __syncthreads();
  if (threadIdx.x < nr) {
    const int r = threadIdx.x;
    float ss = 0.0f;
    for (int g = 0; g < G; ++g) {
      float v[8];
      bf16x8_to_f32(stage[r * pitch + g], v);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = __fadd_rn(ss, __fmul_rn(v[i], v[i]));
    }
    den[r] = norm_den(ss);
    long long q = r0 + r;
    if (padded) {
      const int w = static_cast<int>(q % W);
      q /= W;
      const int h = static_cast<int>(q % H);
      q /= H;
      const int t = static_cast<int>(q % T);
      const long long n = q / T;
      q = ((n * (T + 2) + t + 2) * (H + 2) + h + 1) * (W + 2) + w + 1;
    }
    dst_row[r] = q;
  }
  __syncthreads();
  uint16_t* y = static_cast<uint16_t*>(e.y);
  for (int u = threadIdx.x; u < nr * G; u += blockDim.x) {
    const int r = u / G, g = u - r * G;
    float v[8];
    bf16x8_to_f32(stage[r * pitch + g], v);
    const float d = den[r];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = norm_silu1(v[i], d, e.sqrt_c, __ldg(e.gamma + 8 * g + i));
    *reinterpret_cast<uint4*>(y + dst_row[r] * C + 8 * g) = f32_to_bf16x8(v);
  }
}

// Shared memory of one row-staged block, or 0 when R rows do not fit.
size_t norm_rows_smem(int C, int R) {
  const size_t b = (size_t)R * (C / 8 + 1) * 16 + (size_t)(R + (R & 1)) * 4 + (size_t)R * 8;
  return b <= 200 * 1024 ? b : 0;
}

cudaError_t launch_norm_rows(const void* x, long long rows, const EpiParams& e, int T, int H,
                             int W, int padded, cudaStream_t s) {
  int R = kNormRows;
  while (R > 1 && norm_rows_smem(e.Cout, R) == 0) R /= 2;
  const size_t smem = norm_rows_smem(e.Cout, R);
  if (smem == 0) return cudaErrorInvalidValue;
  static int opted_in[kMaxDevices] = {};
  if (smem > 48 * 1024) {
    const cudaError_t err = opt_in_smem(l2norm_silu_rows_kernel, opted_in);
    if (err != cudaSuccess) return err;
  }
  const long long blocks = (rows + R - 1) / R;
  l2norm_silu_rows_kernel<<<static_cast<unsigned>(blocks), 256, smem, s>>>(
      static_cast<const uint16_t*>(x), rows, e, T, H, W, padded, R);
  return cudaGetLastError();
}

cudaError_t launch_l2norm_silu_pad(const void* x, int N, int T, int H, int W, const EpiParams& e,
                                   cudaStream_t s) {
  return launch_norm_rows(x, (long long)N * T * H * W, e, T, H, W, 1, s);
}

// Everything of the padded output and the cache that is not the activations'
// own padded interiors, one 16-byte group of 8 channels per work item:
//   padded [N, Tc + 2, Hc + 2, Wc + 2, C]: zero on every plane's spatial border and
//     on the planes before the P history planes; history plane 2 - P + j takes
//     prev[:, j] when prev is given (else its interior is left alone); plane t >= 2
//     takes activated frame t - 2 when copy_interior (else left alone);
//   cache [N, K, Hc, Wc, C]: slot k holds frame Tc + P - K + k of the sequence
//     [prev..., activated...]; slots that fall on prev are left alone without prev.
// Activated frame (n, t) pixel (h, w) is at act + n a_sn + t a_st + h a_sh + w C.
// Index type I: 32-bit when every work item index fits (no 64-bit divisions).
template <class I>
__global__ void pad_cache_kernel(PadCacheArgs a) {
  const I G = static_cast<I>(a.C >> 3);
  const I Tp = a.Tc + 2, Hp = a.Hc + 2, Wp = a.Wc + 2;
  const I Hc = a.Hc, Wc = a.Wc, K = a.K;
  const I n_pad = static_cast<I>(a.N) * Tp * Hp * Wp * G;
  const I n_all = n_pad + static_cast<I>(a.N) * K * Hc * Wc * G;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  auto act_at = [&](long long n, int t, int h, int w, int g) {
    return *reinterpret_cast<const uint4*>(a.act + n * a.a_sn + t * a.a_st + h * a.a_sh +
                                           (long long)w * a.C + 8 * g);
  };
  auto prev_at = [&](long long n, int t, int h, int w, int g) {
    return *reinterpret_cast<const uint4*>(
        a.prev + (((n * a.P + t) * a.Hc + h) * a.Wc + w) * a.C + 8 * g);
  };
  const I step = static_cast<I>(gridDim.x) * blockDim.x;
  for (I i = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_all; i += step) {
    if (i < n_pad) {
      I q = i;
      const int g = static_cast<int>(q % G);
      q /= G;
      const int wp = static_cast<int>(q % Wp);
      q /= Wp;
      const int hp = static_cast<int>(q % Hp);
      q /= Hp;
      const int tp = static_cast<int>(q % Tp);
      const long long n = static_cast<long long>(q / Tp);
      uint4* dst = reinterpret_cast<uint4*>(a.padded) + i;
      if (hp == 0 || hp == Hp - 1 || wp == 0 || wp == Wp - 1 || tp < 2 - a.P) {
        *dst = zero;
      } else if (tp >= 2) {
        if (a.copy_interior) *dst = act_at(n, tp - 2, hp - 1, wp - 1, g);
      } else if (a.prev) {
        *dst = prev_at(n, tp - (2 - a.P), hp - 1, wp - 1, g);
      }
    } else {
      const I j = i - n_pad;
      I q = j;
      const int g = static_cast<int>(q % G);
      q /= G;
      const int w = static_cast<int>(q % Wc);
      q /= Wc;
      const int h = static_cast<int>(q % Hc);
      q /= Hc;
      const int k = static_cast<int>(q % K);
      const long long n = static_cast<long long>(q / K);
      const int sidx = a.Tc + a.P - a.K + k;  // position in [prev..., activated...]
      uint4* dst = reinterpret_cast<uint4*>(a.cache) + j;
      if (sidx >= a.P)
        *dst = act_at(n, sidx - a.P, h, w, g);
      else if (a.prev)
        *dst = prev_at(n, sidx, h, w, g);
    }
  }
}

// One item per pixel of the padded input (all Cp channels, 16-byte stores) and per pixel
// of the cache (C channels).  Source frame s of the sequence [history..., chunk...]:
// padded frame f holds s = f - 2 + P (a zero plane for s < 0), cache frame k holds
// s = T + P - K + k.  Threads run along W, so each channel's reads of an NCTHW chunk
// with unit W stride are coalesced.
template <class I>
__global__ void causal_pack_kernel(CausalPackArgs a) {
  const I Tp = a.T + 2, Hp = a.H + 2, Wp = a.W + 2;
  const I n_pad = static_cast<I>(a.N) * Tp * Hp * Wp;
  const I n_all = n_pad + static_cast<I>(a.N) * a.K * a.H * a.W;
  auto src = [&](long long n, int s, int h, int w, int c) -> uint32_t {
    if (s < a.P) return a.prev[(((n * a.P + s) * a.H + h) * a.W + w) * a.C + c];
    return a.x[n * a.sx_n + c * a.sx_c + (s - a.P) * a.sx_t + h * a.sx_h + w * a.sx_w];
  };
  const I step = static_cast<I>(gridDim.x) * blockDim.x;
  for (I i = static_cast<I>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_all; i += step) {
    if (i < n_pad) {
      I q = i;
      const int wp = static_cast<int>(q % Wp);
      q /= Wp;
      const int hp = static_cast<int>(q % Hp);
      q /= Hp;
      const int tp = static_cast<int>(q % Tp);
      const long long n = static_cast<long long>(q / Tp);
      const int s = tp - 2 + a.P;
      const bool zero = hp == 0 || hp == Hp - 1 || wp == 0 || wp == Wp - 1 || s < 0;
      uint16_t* dst = a.padded + static_cast<long long>(i) * a.Cp;
      for (int g = 0; g < a.Cp; g += 8) {
        uint32_t v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = g + 2 * e;
          const uint32_t lo = (!zero && c < a.C) ? src(n, s, hp - 1, wp - 1, c) : 0u;
          const uint32_t hi = (!zero && c + 1 < a.C) ? src(n, s, hp - 1, wp - 1, c + 1) : 0u;
          v[e] = lo | (hi << 16);
        }
        *reinterpret_cast<uint4*>(dst + g) = make_uint4(v[0], v[1], v[2], v[3]);
      }
    } else {
      I q = i - n_pad;
      uint16_t* dst = a.cache + static_cast<long long>(q) * a.C;
      const int w = static_cast<int>(q % a.W);
      q /= a.W;
      const int h = static_cast<int>(q % a.H);
      q /= a.H;
      const int k = static_cast<int>(q % a.K);
      const long long n = static_cast<long long>(q / a.K);
      const int s = a.T + a.P - a.K + k;
      for (int c = 0; c < a.C; ++c) dst[c] = static_cast<uint16_t>(src(n, s, h, w, c));
    }
  }
}

cudaError_t launch_causal_pack(const CausalPackArgs& a, cudaStream_t s) {
  const long long total = (long long)a.N * (a.T + 2) * (a.H + 2) * (a.W + 2) +
                          (long long)a.N * a.K * a.H * a.W;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  if (total + (long long)blocks * threads < 0xFFFFFFFFLL)
    causal_pack_kernel<uint32_t><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
  else
    causal_pack_kernel<unsigned long long><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_pad_cache(const PadCacheArgs& a, cudaStream_t s) {
  const long long G = a.C / 8;
  const long long total = (long long)a.N * (a.Tc + 2) * (a.Hc + 2) * (a.Wc + 2) * G +
                          (long long)a.N * a.K * a.Hc * a.Wc * G;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  if (blocks > 152LL * 16) blocks = 152LL * 16;
  if (blocks < 1) blocks = 1;
  // 32-bit indices while every item index (and the last grid stride past it) fits
  if (total + (long long)blocks * threads < 0xFFFFFFFFLL)
    pad_cache_kernel<uint32_t><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
  else
    pad_cache_kernel<unsigned long long><<<static_cast<unsigned>(blocks), threads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vvc
