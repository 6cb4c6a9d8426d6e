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
cudaError_t launch_l2norm_silu_pad(const void* x, int N, int T, int H, int W, const EpiParams& e,
                                   cudaStream_t s);

}  // namespace vvc
