// Channels-last GroupNorm (+ SiLU): launch arguments shared by the C ABI and the
// kernels in group_norm.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace vvc {

struct GroupNormArgs {
  const uint16_t* x;   // bf16 NDHWC, `slices` x P positions x C channels
  uint16_t* y;         // same shape
  const float* gamma;  // [C] or NULL (1)
  const float* beta;   // [C] or NULL (0)
  double2* partial;    // [slices][chunks][groups] (sum, sum of squares)
  long long P;         // positions per slice: H*W (time-isolated) or D*H*W
  long long chunk;     // positions per block
  int slices, chunks, C, groups, silu;
  float eps;
};

void group_norm_geometry(int C, long long P, int* threads, long long* chunk, int* chunks);
cudaError_t launch_group_norm(const GroupNormArgs& a, int threads, cudaStream_t s);

}  // namespace vvc
