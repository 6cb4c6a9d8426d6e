// Channels-last GroupNorm (+ SiLU) on NDHWC bf16 tensors.
//
// ROCm/FlyDSL issue "[Feature]: conv3d_implicit — accept and emit NDHWC ...",
// MiniMax-H3 comment (section "An extra argument for NDHWC"): every pair of the
// encoder's convolutions is separated by a GroupNorm (+ SiLU) whose groups are
// time-isolated, which NCDHW code reaches only through a time-to-batch copy; in
// NDHWC the frames are already contiguous slices and a group's C / groups channels
// are contiguous at each position, so the reduction reads the tensor in order.
//
// A slice is one frame (n, d) when time_isolated, else one clip n; it is P
// consecutive positions of C channels.  Two launches:
//   1. statistics: a block takes a chunk of a slice's positions; thread t owns the
//      8-channel vector t % V (V = C / 8) of positions t / V, t / V + k, ... (k = block
//      size / V) and sums x and x^2 in fp32; the block folds them per group and
//      writes one fp64 (sum, sum of squares) partial per (slice, chunk, group);
//   2. normalise: each block adds its slice's partials in chunk order in fp64
//      (mean, biased variance, rstd = 1 / sqrt(var + eps)) and writes
//      g = B((x - mean) * rstd * gamma + beta), and with the SiLU B(g / (1 + exp(-g))),
//      8 channels per 16-byte access.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "group_norm.h"

namespace vvc {

namespace {

constexpr int kGnPositionsPerThread = 32;

__device__ __forceinline__ float gn_bf16(float f) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(f)))
                         << 16);
}

__device__ __forceinline__ void gn_unpack(const uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void gn_stats_kernel(GroupNormArgs a) {
  __shared__ float part[2][256][8];
  const int V = a.C >> 3;
  const int k = blockDim.x / V;  // positions in flight per step (blockDim = k V)
  const int t = threadIdx.x;
  const int slice = blockIdx.y;
  const long long p0 = (long long)blockIdx.x * a.chunk;
  const long long p1 = p0 + a.chunk < a.P ? p0 + a.chunk : a.P;
  float s[8], q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) s[i] = q[i] = 0.0f;
  if (t < k * V) {
    const int v = t % V;
    const uint16_t* base = a.x + (long long)slice * a.P * a.C + 8 * v;
    for (long long p = p0 + t / V; p < p1; p += k) {
      float f[8];
      gn_unpack(*reinterpret_cast<const uint4*>(base + p * a.C), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        s[i] += f[i];
        q[i] = fmaf(f[i], f[i], q[i]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    part[0][t][i] = s[i];
    part[1][t][i] = q[i];
  }
  __syncthreads();
  // one thread per group folds the channels of its group over the k position rows
  const int cg = a.C / a.groups;
  for (int g = t; g < a.groups; g += blockDim.x) {
    double S = 0.0, Q = 0.0;
    for (int c = g * cg; c < (g + 1) * cg; ++c) {
      const int v = c >> 3, i = c & 7;
      for (int r = 0; r < k; ++r) {
        S += part[0][r * V + v][i];
        Q += part[1][r * V + v][i];
      }
    }
    double2* out = a.partial + ((long long)slice * a.chunks + blockIdx.x) * a.groups + g;
    *out = make_double2(S, Q);
  }
}

__global__ void gn_norm_kernel(GroupNormArgs a) {
  extern __shared__ float gn_smem[];
  float* mean_c = gn_smem;           // [C] group mean of each channel
  float* scale_c = gn_smem + a.C;    // [C] rstd * gamma
  float* shift_c = gn_smem + 2 * a.C;  // [C] beta
  float* grp = gn_smem + 3 * a.C;    // [2 * groups] mean, rstd
  const int slice = blockIdx.y;
  const double n = (double)a.P * (a.C / a.groups);
  for (int g = threadIdx.x; g < a.groups; g += blockDim.x) {
    double S = 0.0, Q = 0.0;
    const double2* pp = a.partial + (long long)slice * a.chunks * a.groups + g;
    for (int ch = 0; ch < a.chunks; ++ch) {
      const double2 v = pp[(long long)ch * a.groups];
      S += v.x;
      Q += v.y;
    }
    const double mean = S / n;
    double var = Q / n - mean * mean;
    if (var < 0.0) var = 0.0;
    grp[2 * g] = static_cast<float>(mean);
    grp[2 * g + 1] = static_cast<float>(1.0 / sqrt(var + (double)a.eps));
  }
  __syncthreads();
  const int cg = a.C / a.groups;
  for (int c = threadIdx.x; c < a.C; c += blockDim.x) {
    const int g = c / cg;
    mean_c[c] = grp[2 * g];
    scale_c[c] = grp[2 * g + 1] * (a.gamma ? a.gamma[c] : 1.0f);
    shift_c[c] = a.beta ? a.beta[c] : 0.0f;
  }
  __syncthreads();
  // thread t owns the 8 channels of vector t % V at positions t / V, t / V + k, ...
  const int V = a.C >> 3;
  const int k = blockDim.x / V;
  const int t = threadIdx.x;
  if (t >= k * V) return;
  const int v = t % V;
  float m[8], sc[8], sh[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = mean_c[8 * v + i];
    sc[i] = scale_c[8 * v + i];
    sh[i] = shift_c[8 * v + i];
  }
  const long long p0 = (long long)blockIdx.x * a.chunk;
  const long long p1 = p0 + a.chunk < a.P ? p0 + a.chunk : a.P;
  const long long base = (long long)slice * a.P * a.C + 8 * v;
  for (long long p = p0 + t / V; p < p1; p += k) {
    const long long off = base + p * a.C;
    float f[8];
    gn_unpack(*reinterpret_cast<const uint4*>(a.x + off), f);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      float o[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float y = gn_bf16(fmaf(f[i + j] - m[i + j], sc[i + j], sh[i + j]));
        if (a.silu) y = gn_bf16(__fdiv_rn(y, __fadd_rn(1.0f, expf(-y))));
        o[j] = y;
      }
      w[i / 2] = (__float_as_uint(o[0]) >> 16) | (__float_as_uint(o[1]) & 0xFFFF0000u);
    }
    *reinterpret_cast<uint4*>(a.y + off) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

// Positions per chunk and threads per block for C channels (C % 8 == 0, C <= 2048).
void group_norm_geometry(int C, long long P, int* threads, long long* chunk, int* chunks) {
  const int V = C / 8;
  const int k = 256 / V;
  *threads = k * V;
  *chunk = (long long)k * kGnPositionsPerThread;
  *chunks = static_cast<int>((P + *chunk - 1) / *chunk);
}

cudaError_t launch_group_norm(const GroupNormArgs& a, int threads, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(a.chunks), static_cast<unsigned>(a.slices));
  gn_stats_kernel<<<grid, threads, 0, s>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t smem = (size_t)(3 * a.C + 2 * a.groups) * sizeof(float);
  gn_norm_kernel<<<grid, threads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace vvc
