// Small device helpers shared by the tensor-core convolution kernels.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace vvc {

// PyTorch 'reflect' index for a pad of at most L - 1.
__device__ __forceinline__ int reflect_coord(int i, int L) {
  if (i < 0) i = -i;
  if (i >= L) i = 2 * (L - 1) - i;
  return i;
}

// Byte offset under the TMA / UMMA 128B, 64B or 32B swizzle (descriptor layout
// code 2, 4 or 6), relative to a base aligned to the pattern period.  The
// hardware applies the pattern to absolute shared-memory address bits.
__device__ __forceinline__ uint32_t swizzle_off(uint32_t off, int swz) {
  const uint32_t mask = (swz == 2) ? 7u : (swz == 4) ? 3u : 1u;
  return off ^ (((off >> 7) & mask) << 4);
}

__device__ __forceinline__ int swz_code_for_rowbytes(int row_bytes) {
  return row_bytes == 128 ? 2 : (row_bytes == 64 ? 4 : 6);
}

// Bounded wait that ignores the abort flag (used while draining).
__device__ __forceinline__ bool wait_no_abort(uint32_t bar, uint32_t parity,
                                              unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Copies one K-major row of `row_bytes` inside a swizzled operand tile: used to
// write the reflected column of a reflect-padded input row.
__device__ __forceinline__ void copy_swizzled_row(uint8_t* tile, int src_row, int dst_row,
                                                  int row_bytes, int chunk, int swz) {
  const uint32_t so = swizzle_off(static_cast<uint32_t>(src_row * row_bytes + chunk * 16), swz);
  const uint32_t dof = swizzle_off(static_cast<uint32_t>(dst_row * row_bytes + chunk * 16), swz);
  *reinterpret_cast<uint4*>(tile + dof) = *reinterpret_cast<const uint4*>(tile + so);
}

}  // namespace vvc
