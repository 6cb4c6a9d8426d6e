// Channel-major implicit-GEMM convolution with e4m3 operands (ConvCMParams::f8):
// the plain and reflect-W instances, with and without an output halo, compiled
// apart from the bf16 ones so that the units build in parallel.
#include "conv_cm_kernel.cuh"

namespace vvc {

cudaError_t conv_cm_f8_status_read_clear(int* status) {
  int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_conv_cm_status, sizeof(int));
  if (err != cudaSuccess) return err;
  *status = v;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_conv_cm_status, &zero, sizeof(int));
}

// inner: reflect-W halo stages with the inner W taps first (as launch_conv_cm decides).
cudaError_t launch_conv_cm_f8(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                              const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                              const CmHalfMaps& half, const ConvCMParams& p, bool inner,
                              int grid, size_t smem_bytes, cudaStream_t stream) {
  using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CmOutMaps, CmHalfMaps,
                          ConvCMParams);
  if (!p.f8 || p.pair || p.pm || p.gather || p.up2) return cudaErrorInvalidValue;
  const Kernel kernels[4] = {conv_cm_kernel<false, false, false, false, false, false, true>,
                             conv_cm_kernel<false, true, false, false, false, false, true>,
                             conv_cm_kernel<false, false, false, false, true, false, true>,
                             conv_cm_kernel<false, true, false, false, true, false, true>};
  const int which = (p.epi.halo ? 2 : 0) + (inner ? 1 : 0);
  static int opted_in[4][kMaxDevices] = {};
  cudaError_t err = opt_in_smem(kernels[which], opted_in[which]);
  if (err != cudaSuccess) return err;
  kernels[which]<<<grid, 128 + 128 * p.epi_groups, smem_bytes, stream>>>(tmAct, tmWgt, tmWgtLast,
                                                                         om, half, p);
  return cudaGetLastError();
}

}  // namespace vvc
