// Padded output and two-frame cache of the norm + padding variants (cuDNN
// frontend doc "Fused Conv3D + Bias + Residual + RMSNorm + SiLU", sections
// "Normalization and Padding Variant" and "Standalone Normalization and Padding
// Variant"): arguments of the kernel that writes everything except the
// activations' own padded interiors.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace vvc {

struct PadCacheArgs {
  const uint16_t* act;          // activated frames: (n, t, h, w) at act + n a_sn + t a_st
  long long a_sn, a_st, a_sh;   //   + h a_sh + w C (elements)
  const uint16_t* prev;         // NULL, or [N, P, Hc, Wc, C] prior activated frames
  uint16_t* padded;             // [N, Tc + 2, Hc + 2, Wc + 2, C]
  uint16_t* cache;              // [N, K, Hc, Wc, C], K = min(2, Tc + P)
  int N, Tc, Hc, Wc, C;         // C % 8 == 0; every pointer 16-byte aligned
  int P, K;
  int copy_interior;            // 1: write the activations into planes 2 .. Tc + 1
};

cudaError_t launch_pad_cache(const PadCacheArgs& a, cudaStream_t s);

// Input packing of the streaming causal convolution (cuDNN frontend doc, section
// "Causal Conv3D with Cache"): the chunk's frames after up to two history frames, a
// zero causal plane for each missing one, a one-pixel zero border and the channels
// padded to Cp, channels-last; and the chunk's raw history for the next call.
struct CausalPackArgs {
  const uint16_t* x;                   // chunk [N, C, T, H, W] at element strides:
  long long sx_n, sx_c, sx_t, sx_h, sx_w;
  const uint16_t* prev;                // NULL, or [N, P, H, W, C] raw history frames
  uint16_t* padded;                    // [N, T + 2, H + 2, W + 2, Cp]
  uint16_t* cache;                     // [N, K, H, W, C], K = min(2, T + P)
  int N, C, Cp, T, H, W, P, K;         // Cp % 8 == 0, C <= Cp
};

cudaError_t launch_causal_pack(const CausalPackArgs& a, cudaStream_t s);
cudaError_t launch_l2norm_silu_pad(const void* x, int N, int T, int H, int W, const EpiParams& e,
                                   cudaStream_t s);

}  // namespace vvc
