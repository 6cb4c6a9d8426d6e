// Channel-major implicit-GEMM convolution: the instances without an output halo,
// the launcher for every instance, and the status word of this translation unit.
// The kernel itself is in conv_cm_kernel.cuh; the instances that write a haloed
// output are compiled in conv_cm_halo.cu, the e4m3 ones in conv_cm_f8.cu.
#include "conv_cm_kernel.cuh"

namespace vvc {

cudaError_t launch_conv_cm_halo(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                                const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                                const CmHalfMaps& half, const ConvCMParams& p, int which,
                                int grid, size_t smem_bytes, cudaStream_t stream);
cudaError_t conv_cm_halo_status_read_clear(int* status);
cudaError_t launch_conv_cm_f8(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                              const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                              const CmHalfMaps& half, const ConvCMParams& p, bool inner,
                              int grid, size_t smem_bytes, cudaStream_t stream);
cudaError_t conv_cm_f8_status_read_clear(int* status);

cudaError_t conv_cm_status_read_clear(int* status) {
  int v = 0;
  cudaError_t err = cudaMemcpyFromSymbol(&v, g_conv_cm_status, sizeof(int));
  if (err != cudaSuccess) return err;
  const int zero = 0;
  err = cudaMemcpyToSymbol(g_conv_cm_status, &zero, sizeof(int));
  if (err != cudaSuccess) return err;
  int h = 0, f = 0;
  err = conv_cm_halo_status_read_clear(&h);
  if (err != cudaSuccess) return err;
  err = conv_cm_f8_status_read_clear(&f);
  if (err != cudaSuccess) return err;
  *status = v ? v : (h ? h : f);
  return cudaSuccess;
}

cudaError_t launch_conv_cm(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                           const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                           const CmHalfMaps& half, const ConvCMParams& p, int grid,
                           size_t smem_bytes, cudaStream_t stream) {
  // the same condition as the MMA warp's reflect-W handling in the plain instance
  const bool inner = p.reflect_w && p.halo && !p.pm && p.KS >= 3;
  // the plan never pairs reflect-W or pixel-major layers
  if (p.pair && (inner || p.pm)) return cudaErrorInvalidValue;
  if (p.gather && (p.pair || p.pm)) return cudaErrorInvalidValue;
  if (p.up2 && (p.pair || p.pm || p.gather || inner || p.epi.halo || !p.halo))
    return cudaErrorInvalidValue;
  if (p.f8)
    return launch_conv_cm_f8(tmAct, tmWgt, tmWgtLast, om, half, p, inner, grid, smem_bytes,
                             stream);
  const int which = p.up2 ? 5 : (p.gather ? 4 : (p.pm ? 3 : (p.pair ? 1 : (inner ? 2 : 0))));
  if (p.epi.halo)
    return launch_conv_cm_halo(tmAct, tmWgt, tmWgtLast, om, half, p, which, grid, smem_bytes,
                               stream);
  using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CmOutMaps, CmHalfMaps,
                          ConvCMParams);
  const Kernel kernels[6] = {conv_cm_kernel<false, false, false, false, false, false>,
                             conv_cm_kernel<true, false, false, false, false, false>,
                             conv_cm_kernel<false, true, false, false, false, false>,
                             conv_cm_kernel<false, false, true, false, false, false>,
                             conv_cm_kernel<false, false, false, true, false, false>,
                             conv_cm_kernel<false, false, false, false, false, true>};
  static int opted_in[6][kMaxDevices] = {};
  cudaError_t err = opt_in_smem(kernels[which], opted_in[which]);
  if (err != cudaSuccess) return err;
  kernels[which]<<<grid, 128 + 128 * p.epi_groups, smem_bytes, stream>>>(tmAct, tmWgt, tmWgtLast,
                                                                         om, half, p);
  return cudaGetLastError();
}

}  // namespace vvc
