// Channel-major implicit-GEMM convolution: the instances that write their output
// inside a haloed tensor (EpiParams::halo; the next call of a chain reads it as a
// padded input), compiled apart from the others so that both build in parallel.
#include "conv_cm_kernel.cuh"

namespace vvc {

cudaError_t conv_cm_halo_status_read_clear(int* status) {
  int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_conv_cm_status, sizeof(int));
  if (err != cudaSuccess) return err;
  *status = v;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_conv_cm_status, &zero, sizeof(int));
}

// which: 0 plain, 1 paired last chunks, 2 reflect-W inner taps first, 3 pixel-major,
// 4 narrow-input gather (as launch_conv_cm numbers them).
cudaError_t launch_conv_cm_halo(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                                const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                                const CmHalfMaps& half, const ConvCMParams& p, int which,
                                int grid, size_t smem_bytes, cudaStream_t stream) {
  using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CmOutMaps, CmHalfMaps,
                          ConvCMParams);
  if (which < 0 || which > 4) return cudaErrorInvalidValue;
  const Kernel kernels[5] = {conv_cm_kernel<false, false, false, false, true, false>,
                             conv_cm_kernel<true, false, false, false, true, false>,
                             conv_cm_kernel<false, true, false, false, true, false>,
                             conv_cm_kernel<false, false, true, false, true, false>,
                             conv_cm_kernel<false, false, false, true, true, false>};
  static int opted_in[5][kMaxDevices] = {};
  cudaError_t err = opt_in_smem(kernels[which], opted_in[which]);
  if (err != cudaSuccess) return err;
  kernels[which]<<<grid, 128 + 128 * p.epi_groups, smem_bytes, stream>>>(tmAct, tmWgt, tmWgtLast,
                                                                         om, half, p);
  return cudaGetLastError();
}

}  // namespace vvc
