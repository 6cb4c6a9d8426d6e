// ORACLE — test infrastructure only.
//
// A plain, slow CPU restatement of what the video-VAE convolution path
// computes, used to check the CUDA library.  Only the tests, the smoke check
// and the benchmark's CPU-baseline leg may load this library; the product path
// never does.  It shares no code, header or constant with the CUDA sources.
//
// Sources followed (web pages, cited by title and section):
//  [FlyDSL#993]  ROCm/FlyDSL issue "[Feature]: conv3d_implicit — accept and
//                emit NDHWC so chained convs skip the layout round-trip".
//  [FlyDSL#1069] ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv
//                shapes to conv3d tests".
//  [cuDNN-PO]    cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm
//                + SiLU".
//
// Every routine is the plain definition: no blocking, no fusion, no
// reordering beyond what the definition states.  Accumulation is in double
// (exact for bf16*bf16 products at these sizes), then rounded to fp32 once,
// matching "Convolution accumulates in FP32" ([cuDNN-PO], Operation Contract)
// up to summation order.
//
// Parity pins (see tests/test_oracle_*.py): brute force against an explicit
// pad + 7-loop convolution written separately in numpy, torch fp64 conv3d,
// the T=1 causal identity ([FlyDSL#1069], "T=1 degeneration"), 1x1x1 == GEMM,
// layout round trip, closed forms (ones, one-hot, stride subsampling) and the
// post-norm row-norm invariant.  Summation order inside the GPU mainloop is
// the one part left free ("parity unpinned" beyond +-1 bf16 ulp of conv).
//
// Compile with -ffp-contract=off: every fp32 operation of the epilogue is a
// separately rounded IEEE operation, as the contract's pseudo-code reads.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

// ---- bf16 <-> fp32 -----------------------------------------------------------
// B(x): fp32 -> bf16 with round-to-nearest-even ([cuDNN-PO], Operation
// Contract, "Let B(x) denote BF16 conversion"; the rounding mode is not stated,
// read as RNE like torch's .to(bfloat16)).  Subnormals are kept.
inline float bf2f(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

inline uint16_t f2bf(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7fffffffu) > 0x7f800000u)  // NaN stays NaN (quiet)
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
  // round half to even on the 16 dropped bits
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
  return static_cast<uint16_t>(upper);
}

inline float B(float f) { return bf2f(f2bf(f)); }

// ---- padded coordinate -> source coordinate ------------------------------------
// zero pad: outside [0, L) reads 0 (returns -1).
// reflect pad: PyTorch 'reflect' (edge not repeated): -i for i < 0 and
// 2(L-1)-i for i >= L.  [FlyDSL#993] describes the VAE's own padding as
// "spatial reflect pad + temporal causal pad", applied before a padding=0 conv.
inline long src_coord(long i, long L, int mode) {
  if (i >= 0 && i < L) return i;
  if (mode == 0) return -1;
  long j = (i < 0) ? -i : 2 * (L - 1) - i;
  if (j < 0 || j >= L) return -2;  // reflect wider than the tensor: invalid
  return j;
}

struct Geo {
  int layout;  // 0 = NCDHW, 1 = NDHWC
  long N, C, D, H, W;
  long Co, KT, KR, KS;
  long st, sh, sw;
  long pb[3], pa[3];
  int pm[3];
  long Do, Ho, Wo;
};

inline long x_index(const Geo& g, long n, long c, long d, long h, long w) {
  if (g.layout == 0) return (((n * g.C + c) * g.D + d) * g.H + h) * g.W + w;
  return (((n * g.D + d) * g.H + h) * g.W + w) * g.C + c;
}

int make_geo(Geo& g, int layout, int N, int C, int D, int H, int W, int Co, int KT,
             int KR, int KS, int st, int sh, int sw, const int* pads) {
  g.layout = layout;
  g.N = N; g.C = C; g.D = D; g.H = H; g.W = W;
  g.Co = Co; g.KT = KT; g.KR = KR; g.KS = KS;
  g.st = st; g.sh = sh; g.sw = sw;
  const long L[3] = {D, H, W};
  for (int k = 0; k < 3; ++k) {
    g.pb[k] = pads[3 * k + 0];
    g.pa[k] = pads[3 * k + 1];
    g.pm[k] = pads[3 * k + 2];
    if (g.pb[k] < 0 || g.pa[k] < 0) return -1;
    if (g.pm[k] == 1 && (g.pb[k] >= L[k] || g.pa[k] >= L[k])) return -1;
  }
  if (N < 1 || C < 1 || D < 1 || H < 1 || W < 1 || Co < 1) return -1;
  if (KT < 1 || KR < 1 || KS < 1 || st < 1 || sh < 1 || sw < 1) return -1;
  g.Do = (D + g.pb[0] + g.pa[0] - KT) / st + 1;
  g.Ho = (H + g.pb[1] + g.pa[1] - KR) / sh + 1;
  g.Wo = (W + g.pb[2] + g.pa[2] - KS) / sw + 1;
  if (D + g.pb[0] + g.pa[0] < KT || H + g.pb[1] + g.pa[1] < KR ||
      W + g.pb[2] + g.pa[2] < KS)
    return -1;
  return 0;
}

// Weight reordered to [t][r][s][ci][co] in double, so the innermost loop over
// output channels is contiguous.  This is only a change of storage order.
std::vector<double> weight_by_tap(const Geo& g, const uint16_t* w) {
  std::vector<double> wt(static_cast<size_t>(g.KT * g.KR * g.KS * g.C * g.Co));
  for (long co = 0; co < g.Co; ++co)
    for (long ci = 0; ci < g.C; ++ci)
      for (long t = 0; t < g.KT; ++t)
        for (long r = 0; r < g.KR; ++r)
          for (long s = 0; s < g.KS; ++s) {
            long src = (((co * g.C + ci) * g.KT + t) * g.KR + r) * g.KS + s;
            long tap = (t * g.KR + r) * g.KS + s;
            wt[static_cast<size_t>((tap * g.C + ci) * g.Co + co)] = bf2f(w[src]);
          }
  return wt;
}

// One output pixel, all output channels:
//   acc[co] = sum_{t,r,s,ci} x[n, ci, od*st+t-pt, oh*sh+r-ph, ow*sw+s-pw] * W[co,ci,t,r,s]
// a cross-correlation like F.conv3d ([FlyDSL#993], "conv3d_implicit";
// [cuDNN-PO], "Raw Conv3D Variant").
void one_pixel(const Geo& g, const uint16_t* x, const std::vector<double>& wt, long n,
               long od, long oh, long ow, double* acc, double* xrow) {
  for (long co = 0; co < g.Co; ++co) acc[co] = 0.0;
  for (long t = 0; t < g.KT; ++t) {
    long id = src_coord(od * g.st + t - g.pb[0], g.D, g.pm[0]);
    if (id < 0) continue;
    for (long r = 0; r < g.KR; ++r) {
      long ih = src_coord(oh * g.sh + r - g.pb[1], g.H, g.pm[1]);
      if (ih < 0) continue;
      for (long s = 0; s < g.KS; ++s) {
        long iw = src_coord(ow * g.sw + s - g.pb[2], g.W, g.pm[2]);
        if (iw < 0) continue;
        for (long ci = 0; ci < g.C; ++ci) xrow[ci] = bf2f(x[x_index(g, n, ci, id, ih, iw)]);
        long tap = (t * g.KR + r) * g.KS + s;
        const double* wtap = wt.data() + tap * g.C * g.Co;
        for (long ci = 0; ci < g.C; ++ci) {
          double xv = xrow[ci];
          if (xv == 0.0) continue;
          const double* wrow = wtap + ci * g.Co;
          for (long co = 0; co < g.Co; ++co) acc[co] += xv * wrow[co];
        }
      }
    }
  }
}

int set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
  return omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

}  // namespace

extern "C" {

int orc_num_threads(int nthreads) { return set_threads(nthreads); }

// Output extent of the convolution: (L + before + after - K) / stride + 1.
int orc_out_dims(int D, int H, int W, int KT, int KR, int KS, int st, int sh, int sw,
                 const int* pads, int* out3) {
  Geo g;
  if (make_geo(g, 1, 1, 1, D, H, W, 1, KT, KR, KS, st, sh, sw, pads) != 0) return -1;
  out3[0] = static_cast<int>(g.Do);
  out3[1] = static_cast<int>(g.Ho);
  out3[2] = static_cast<int>(g.Wo);
  return 0;
}

// Full convolution.  acc_out is fp32 [N][Do][Ho][Wo][Co]: the double sum
// rounded once to fp32.  pads = 9 ints: (before, after, mode) for T, H, W;
// mode 0 = zero, 1 = reflect.  x is bf16 bits in `layout` (0 NCDHW, 1 NDHWC);
// w is bf16 bits in the checkpoint order OITRS.
int orc_conv3d_acc(const uint16_t* x, int layout, int N, int C, int D, int H, int W,
                   const uint16_t* w, int Co, int KT, int KR, int KS, int st, int sh,
                   int sw, const int* pads, float* acc_out, int nthreads) {
  Geo g;
  if (make_geo(g, layout, N, C, D, H, W, Co, KT, KR, KS, st, sh, sw, pads) != 0) return -1;
  set_threads(nthreads);
  std::vector<double> wt = weight_by_tap(g, w);
  const long P = g.N * g.Do * g.Ho * g.Wo;
#pragma omp parallel
  {
    std::vector<double> acc(static_cast<size_t>(g.Co)), xrow(static_cast<size_t>(g.C));
#pragma omp for schedule(dynamic, 16)
    for (long p = 0; p < P; ++p) {
      long ow = p % g.Wo, q = p / g.Wo;
      long oh = q % g.Ho;
      q /= g.Ho;
      long od = q % g.Do, n = q / g.Do;
      one_pixel(g, x, wt, n, od, oh, ow, acc.data(), xrow.data());
      float* dst = acc_out + p * g.Co;
      for (long co = 0; co < g.Co; ++co) dst[co] = static_cast<float>(acc[co]);
    }
  }
  return 0;
}

// Selected output pixels only: points = P x 4 int64 (n, od, oh, ow);
// acc_out = fp32 [P][Co].  Used for sampled checks at full sizes.
int orc_conv3d_acc_points(const uint16_t* x, int layout, int N, int C, int D, int H,
                          int W, const uint16_t* w, int Co, int KT, int KR, int KS, int st,
                          int sh, int sw, const int* pads, const int64_t* points, long P,
                          float* acc_out, int nthreads) {
  Geo g;
  if (make_geo(g, layout, N, C, D, H, W, Co, KT, KR, KS, st, sh, sw, pads) != 0) return -1;
  for (long i = 0; i < P; ++i) {
    const int64_t* pt = points + 4 * i;
    if (pt[0] < 0 || pt[0] >= g.N || pt[1] < 0 || pt[1] >= g.Do || pt[2] < 0 ||
        pt[2] >= g.Ho || pt[3] < 0 || pt[3] >= g.Wo)
      return -2;
  }
  set_threads(nthreads);
  std::vector<double> wt = weight_by_tap(g, w);
#pragma omp parallel
  {
    std::vector<double> acc(static_cast<size_t>(g.Co)), xrow(static_cast<size_t>(g.C));
#pragma omp for schedule(dynamic, 4)
    for (long i = 0; i < P; ++i) {
      const int64_t* pt = points + 4 * i;
      one_pixel(g, x, wt, pt[0], pt[1], pt[2], pt[3], acc.data(), xrow.data());
      float* dst = acc_out + i * g.Co;
      for (long co = 0; co < g.Co; ++co) dst[co] = static_cast<float>(acc[co]);
    }
  }
  return 0;
}

// B(x) elementwise: fp32 -> bf16 bits.
void orc_round_bf16(const float* in, uint16_t* out, long n) {
  for (long i = 0; i < n; ++i) out[i] = f2bf(in[i]);
}

// Epilogue flags (oracle-local numbering).
enum { ORC_BIAS = 1, ORC_RESIDUAL = 2, ORC_RESIDUAL_BIAS = 4, ORC_L2NORM_SILU = 8 };

// Post-operations on rows of `conv` (bf16 bits, [M][C], one row per output
// pixel), exactly as [cuDNN-PO], Operation Contract:
//   main  = B(conv + bias)                      (main = conv without bias)
//   skip  = residual, or B(residual + residual_bias)
//   value = B(main + skip)                      (value = main without residual)
//   den   = max(sqrt(sum_c value_c^2), 1e-12)   (serial fp32 sum over the row)
//   normalized = B(value / den); scaled = B(normalized * sqrt(C))
//   affine = B(scaled * gamma); activated = B(affine / (1 + exp(-affine)))
// main_out / value_out / act_out may be null.  act_out needs ORC_L2NORM_SILU.
int orc_epilogue(const uint16_t* conv, long M, int C, unsigned flags, const float* bias,
                 const uint16_t* residual, const float* residual_bias, const float* gamma,
                 uint16_t* main_out, uint16_t* value_out, uint16_t* act_out, int nthreads) {
  if ((flags & ORC_RESIDUAL_BIAS) && !(flags & ORC_RESIDUAL)) return -1;
  if ((flags & ORC_L2NORM_SILU) && !gamma) return -1;
  if ((flags & ORC_BIAS) && !bias) return -1;
  if ((flags & ORC_RESIDUAL) && !residual) return -1;
  if ((flags & ORC_RESIDUAL_BIAS) && !residual_bias) return -1;
  set_threads(nthreads);
  const float sqrt_c = std::sqrt(static_cast<float>(C));
#pragma omp parallel
  {
    std::vector<float> value(static_cast<size_t>(C));
#pragma omp for schedule(static)
    for (long m = 0; m < M; ++m) {
      for (int c = 0; c < C; ++c) {
        long i = m * C + c;
        float mainv = bf2f(conv[i]);
        if (flags & ORC_BIAS) mainv = B(mainv + bias[c]);
        if (main_out) main_out[i] = f2bf(mainv);
        float v = mainv;
        if (flags & ORC_RESIDUAL) {
          float skip = bf2f(residual[i]);
          if (flags & ORC_RESIDUAL_BIAS) skip = B(skip + residual_bias[c]);
          v = B(mainv + skip);
        }
        value[static_cast<size_t>(c)] = v;
        if (value_out) value_out[i] = f2bf(v);
      }
      if (flags & ORC_L2NORM_SILU) {
        float ss = 0.0f;
        for (int c = 0; c < C; ++c) {
          float sq = value[static_cast<size_t>(c)] * value[static_cast<size_t>(c)];
          ss = ss + sq;
        }
        float den = std::sqrt(ss);
        if (!(den > 1e-12f)) den = 1e-12f;  // max(norm, 1e-12)
        for (int c = 0; c < C; ++c) {
          float nrm = B(value[static_cast<size_t>(c)] / den);
          float sc = B(nrm * sqrt_c);
          float af = B(sc * gamma[c]);
          float e = std::exp(-af);
          float act = B(af / (1.0f + e));
          if (act_out) act_out[m * C + c] = f2bf(act);
        }
      }
    }
  }
  return 0;
}

// Standalone post-operations on an existing bf16 tensor [rows][C] without a
// convolution ([cuDNN-PO], "Standalone Normalization and Padding Variant"):
// main = B(raw + input_bias) when input_bias is given, else raw; then the same
// residual / norm / SiLU steps as orc_epilogue.
int orc_l2norm_silu(const uint16_t* raw, long rows, int C, const float* input_bias,
                    const uint16_t* residual, const float* residual_bias,
                    const float* gamma, uint16_t* y, uint16_t* value_out, int nthreads) {
  unsigned flags = ORC_L2NORM_SILU;
  if (input_bias) flags |= ORC_BIAS;
  if (residual) flags |= ORC_RESIDUAL;
  if (residual_bias) flags |= ORC_RESIDUAL_BIAS;
  return orc_epilogue(raw, rows, C, flags, input_bias, residual, residual_bias, gamma,
                      nullptr, value_out, y, nthreads);
}

// Weight pack ([cuDNN-PO], "Weight Packing"): OITRS -> OTRSI, each
// input-channel row zero-padded to a multiple of 64.
int orc_pack_weight(const uint16_t* w, int Co, int Ci, int KT, int KR, int KS,
                    uint16_t* packed) {
  if (Co < 1 || Ci < 1 || KT < 1 || KR < 1 || KS < 1) return -1;
  const long cp = (static_cast<long>(Ci) + 63) / 64 * 64;
  for (long co = 0; co < Co; ++co)
    for (long t = 0; t < KT; ++t)
      for (long r = 0; r < KR; ++r)
        for (long s = 0; s < KS; ++s)
          for (long ci = 0; ci < cp; ++ci) {
            long dst = (((co * KT + t) * KR + r) * KS + s) * cp + ci;
            packed[dst] = (ci < Ci) ? w[(((co * Ci + ci) * KT + t) * KR + r) * KS + s] : 0;
          }
  return 0;
}

}  // extern "C"
