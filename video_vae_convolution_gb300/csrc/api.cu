// C ABI of the convolution library: argument validation, the launch plan
// (input staging, tile shape, pipeline depth, split of the reduction), TMA
// tensor-map encoding and kernel dispatch.  See include/conv3d.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "conv3d.h"
#include "internal.h"
#include "group_norm.h"
#include "pad_cache.h"

namespace vvc {
cudaError_t launch_conv_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const ConvTCParams& p,
                           dim3 grid, size_t smem_bytes, cudaStream_t stream);
cudaError_t launch_conv_cm(const CUtensorMap& tmAct, const CUtensorMap& tmWgt,
                           const CUtensorMap& tmWgtLast, const CmOutMaps& om,
                           const CmHalfMaps& half, const ConvCMParams& p, int grid,
                           size_t smem_bytes, cudaStream_t stream);
cudaError_t conv_status_read_clear(int* status, cudaStream_t stream);
cudaError_t conv_cm_status_read_clear(int* status);
cudaError_t launch_pack_weight_u8(const void* w, void* out, int Co, int Ci, int taps,
                                  cudaStream_t s);
cudaError_t launch_pack_weight(const void* w, void* out, int Co, int Ci, int taps,
                               cudaStream_t s);
cudaError_t launch_stage_input(const void* x, int layout, int N, int C, int Cp, long long S,
                               void* out, cudaStream_t s);
cudaError_t launch_im2col_hw(const void* x, int layout, int N, int C, int D, int H, int W, int Ho,
                             int Wo, int KT, int KR, int KS, int sh, int sw, int ph, int pw,
                             int reflect_h, int reflect_w, int Ck, void* out, const void* wp,
                             int Cout, void* wr, cudaStream_t s);
cudaError_t launch_splitk_epilogue(const float* partial, int splits, long long M,
                                   const EpiParams& e, cudaStream_t s);
cudaError_t launch_l2norm_silu(const void* x, long long rows, const EpiParams& e,
                               cudaStream_t s);
}  // namespace vvc

namespace {

using vvc::ConvCMParams;
using vvc::ConvTCParams;
using vvc::EpiParams;

constexpr size_t kMaxSmem = 232448;  // sm_100 / sm_103 opt-in dynamic shared memory per block
constexpr int kDefaultSMs = 152;  // GB300
// Per-warp epilogue staging block of the channel-major kernel (kStageFloats fp32).
constexpr size_t kEpiWarpBytes = 32 * 36 * 4;

// SM count of the current device (cached per device; 152 when there is none).
int num_sms() {
  static int cached[vvc::kMaxDevices] = {};
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vvc::kMaxDevices) {
    (void)cudaGetLastError();
    return kDefaultSMs;
  }
  const int c = __atomic_load_n(&cached[dev], __ATOMIC_RELAXED);
  if (c) return c;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = kDefaultSMs;
  }
  __atomic_store_n(&cached[dev], n, __ATOMIC_RELAXED);
  return n;
}

inline long long round_up(long long a, long long b) { return (a + b - 1) / b * b; }

// Limit of every device-side wait: 4 s, or CONV3D_TIMEOUT_MS from the environment
// (read once; lets a test run fail fast).
int default_timeout_ms() {
  static int ms = -1;
  if (ms < 0) {
    const char* e = std::getenv("CONV3D_TIMEOUT_MS");
    const int v = e ? std::atoi(e) : 0;
    ms = (v > 0) ? v : 4000;
  }
  return ms;
}
inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

struct Plan {
  int Do = 0, Ho = 0, Wo = 0;
  bool stage = false;
  int Cst = 0;
  size_t stage_off = 0, stage_bytes = 0;
  size_t partial_off = 0, partial_bytes = 0;
  size_t vscratch_off = 0, vscratch_bytes = 0;
  size_t ws_bytes = 0;
  // narrow input: the staging kernel gathers the spatial taps (im2col) and the
  // convolution runs as (KT, 1, 1) over Ck channels with repacked weights
  bool im2col = false;
  int Ck = 0;
  size_t wr_off = 0, wr_bytes = 0;
  conv3d_params q{};
  // e4m3 operands: the kernels see a bf16-sized convolution over channel pairs (q)
  bool f8 = false;
  bool cm = false;          // channel-major kernel (conv_cm) instead of pixel-major (conv_tc)
  ConvTCParams kp{};
  ConvCMParams cp{};
  dim3 grid;
  size_t smem = 0;
  int launches = 0;
  // padded output + cache: the kernels write the activations to a contiguous
  // [N, Do, Ho, Wo, Cout] scratch buffer at pc_off, and one more launch places them
  bool pad_cache = false;
  size_t pc_off = 0, pc_bytes = 0;
};

struct Span {
  uintptr_t lo, hi;
};

bool overlaps(const Span& a, const Span& b) {
  return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo;
}

int out_extent(int L, int b, int a, int K, int s) {
  const long long num = (long long)L + b + a - K;
  if (num < 0) return -1;
  return static_cast<int>(num / s + 1);
}

bool has_halo(const conv3d_params* p) {
  for (int i = 0; i < 3; ++i)
    if (p->out_halo[i].before || p->out_halo[i].after) return true;
  return false;
}

// Extents of y: [N, Do + tb + ta, Ho + hb + ha, Wo + wb + wa] with an output halo.
void y_extent(const conv3d_params* p, int Do, int Ho, int Wo, long long* Dy, long long* Hy,
              long long* Wy) {
  *Dy = (long long)Do + p->out_halo[0].before + p->out_halo[0].after;
  *Hy = (long long)Ho + p->out_halo[1].before + p->out_halo[1].after;
  *Wy = (long long)Wo + p->out_halo[2].before + p->out_halo[2].after;
}

// Geometry and flag validation; no CUDA calls.
int validate_shape(const conv3d_params* p, int* Do, int* Ho, int* Wo) {
  if (!p) return CONV3D_ERR_INVALID_ARG;
  if (p->layout != CONV3D_NCDHW && p->layout != CONV3D_NDHWC) return CONV3D_ERR_INVALID_ARG;
  if (p->out_layout != CONV3D_NCDHW && p->out_layout != CONV3D_NDHWC)
    return CONV3D_ERR_INVALID_ARG;
  if (p->N < 1 || p->Cin < 1 || p->D < 1 || p->H < 1 || p->W < 1 || p->Cout < 1)
    return CONV3D_ERR_INVALID_ARG;
  if (p->KT < 1 || p->KR < 1 || p->KS < 1) return CONV3D_ERR_INVALID_ARG;
  for (int i = 0; i < 3; ++i) {
    if (p->stride[i] < 1) return CONV3D_ERR_INVALID_ARG;
    if (p->pad[i].before < 0 || p->pad[i].after < 0) return CONV3D_ERR_INVALID_ARG;
    if (p->pad[i].mode != CONV3D_PAD_ZERO && p->pad[i].mode != CONV3D_PAD_REFLECT)
      return CONV3D_ERR_INVALID_ARG;
  }
  if (p->input_upsample != 0 && p->input_upsample != 2) return CONV3D_ERR_INVALID_ARG;
  if (p->dtype != CONV3D_DTYPE_BF16 && p->dtype != CONV3D_DTYPE_E4M3) return CONV3D_ERR_INVALID_ARG;
  if (p->dtype == CONV3D_DTYPE_E4M3) {
    // FP8 e4m3 operands: channels-last bytes, 16-byte channel rows, a usable scale
    if (p->layout != CONV3D_NDHWC || p->Cin % 16 != 0 || p->input_upsample != 0 ||
        !std::isfinite(p->fp8_scale) || p->fp8_scale == 0.0f)
      return CONV3D_ERR_INVALID_ARG;
  }
  const int up = p->input_upsample == 2 ? 2 : 1;  // the convolution reads the x2 grid
  if ((long long)p->H * up > 0x3fffffffLL || (long long)p->W * up > 0x3fffffffLL)
    return CONV3D_ERR_INVALID_ARG;
  const int L[3] = {p->D, p->H * up, p->W * up};
  const int K[3] = {p->KT, p->KR, p->KS};
  int o[3];
  for (int i = 0; i < 3; ++i) {
    if (p->pad[i].mode == CONV3D_PAD_REFLECT &&
        (p->pad[i].before >= L[i] || p->pad[i].after >= L[i]))
      return CONV3D_ERR_INVALID_ARG;
    o[i] = out_extent(L[i], p->pad[i].before, p->pad[i].after, K[i], p->stride[i]);
    if (o[i] < 1) return CONV3D_ERR_INVALID_ARG;
  }
  const unsigned e = p->epi;
  const unsigned known = CONV3D_EPI_BIAS | CONV3D_EPI_RESIDUAL | CONV3D_EPI_RESIDUAL_BIAS |
                         CONV3D_EPI_L2NORM_SILU | CONV3D_EPI_SAVE_VALUE |
                         CONV3D_EPI_OUT_PAD_BR | CONV3D_EPI_PAD_CACHE |
                         CONV3D_EPI_DEBUG_STORE_CONV;
  if (e & ~known) return CONV3D_ERR_INVALID_ARG;
  if (e & CONV3D_EPI_PAD_CACHE) {
    // padded output + cache: the activations of the fused norm, channels last
    if (!(e & CONV3D_EPI_L2NORM_SILU) || (e & CONV3D_EPI_OUT_PAD_BR) ||
        p->out_layout != CONV3D_NDHWC || p->Cout % 8 != 0 || p->history_frames < 0 ||
        p->history_frames > 2 || !p->cache_out)
      return CONV3D_ERR_INVALID_ARG;
  }
  if (has_halo(p)) {
    // output halo: NDHWC, 16-byte channel rows, unwritten zero-mode T halo, H / W
    // halos of at most one pixel per side (reflection needs two output pixels)
    const conv3d_pad* hl = p->out_halo;
    if (p->out_layout != CONV3D_NDHWC || p->Cout % 8 != 0 ||
        (e & (CONV3D_EPI_L2NORM_SILU | CONV3D_EPI_OUT_PAD_BR | CONV3D_EPI_PAD_CACHE)) ||
        hl[0].mode != CONV3D_PAD_ZERO || hl[0].before < 0 || hl[0].after < 0)
      return CONV3D_ERR_INVALID_ARG;
    for (int i = 1; i < 3; ++i) {
      if (hl[i].before < 0 || hl[i].before > 1 || hl[i].after < 0 || hl[i].after > 1 ||
          (hl[i].mode != CONV3D_PAD_ZERO && hl[i].mode != CONV3D_PAD_REFLECT))
        return CONV3D_ERR_INVALID_ARG;
      if (hl[i].mode == CONV3D_PAD_REFLECT && o[i] < 2) return CONV3D_ERR_INVALID_ARG;
    }
  }
  if (p->input_upsample == 2) {
    // x2 nearest upsampled input before a 3x3, pad-1, stride-1 (along H and W) conv
    if (p->KR != 3 || p->KS != 3 || p->stride[1] != 1 || p->stride[2] != 1 ||
        p->pad[1].before != 1 || p->pad[1].after != 1 || p->pad[1].mode != CONV3D_PAD_ZERO ||
        p->pad[2].before != 1 || p->pad[2].after != 1 || p->pad[2].mode != CONV3D_PAD_ZERO ||
        p->out_layout != CONV3D_NDHWC || p->Cout % 8 != 0 || has_halo(p) ||
        (e & (CONV3D_EPI_RESIDUAL | CONV3D_EPI_L2NORM_SILU | CONV3D_EPI_SAVE_VALUE |
              CONV3D_EPI_OUT_PAD_BR | CONV3D_EPI_PAD_CACHE)))
      return CONV3D_ERR_INVALID_ARG;
  }
  if ((e & CONV3D_EPI_RESIDUAL_BIAS) && !(e & CONV3D_EPI_RESIDUAL)) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_OUT_PAD_BR) && (e & CONV3D_EPI_L2NORM_SILU)) return CONV3D_ERR_INVALID_ARG;
  if (!p->x || !p->w_packed || !p->y) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_BIAS) && !p->bias) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_RESIDUAL) && !p->residual) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_RESIDUAL_BIAS) && !p->residual_bias) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_L2NORM_SILU) && !p->gamma) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_SAVE_VALUE) && !p->value_out) return CONV3D_ERR_INVALID_ARG;
  if ((e & CONV3D_EPI_DEBUG_STORE_CONV) && !p->conv_out) return CONV3D_ERR_INVALID_ARG;
  // element counts must stay addressable with 32-bit TMA coordinates
  if ((long long)p->KT * p->KR * p->KS * round_up(p->Cin, 64) > 0x7fffffffLL)
    return CONV3D_ERR_UNSUPPORTED;
  *Do = o[0];
  *Ho = o[1];
  *Wo = o[2];
  return CONV3D_OK;
}

// Covered by the kernels (beyond plain validity).
int check_supported(const conv3d_params* p) {
  if (p->pad[0].mode == CONV3D_PAD_REFLECT && (p->pad[0].before || p->pad[0].after))
    return CONV3D_ERR_UNSUPPORTED;  // reflect along T: not used by the VAE paths
  if (p->pad[2].mode == CONV3D_PAD_REFLECT) {
    if (p->pad[2].before > 1 || p->pad[2].after > 1) return CONV3D_ERR_UNSUPPORTED;
    if (p->stride[2] > 2) return CONV3D_ERR_UNSUPPORTED;
    if (p->W < 3) return CONV3D_ERR_UNSUPPORTED;
  }
  if (p->KS > 8 || p->KR > 64 || p->KT > 64) return CONV3D_ERR_UNSUPPORTED;
  if ((p->epi & CONV3D_EPI_L2NORM_SILU) && p->Cout > 512) return CONV3D_ERR_UNSUPPORTED;
  if (p->stride[2] > 8) return CONV3D_ERR_UNSUPPORTED;
  return CONV3D_OK;
}

// Epilogue parameters common to both kernels.
void fill_epi(const conv3d_params* p, const Plan& pl, EpiParams* e) {
  e->y = p->y;
  e->out_layout = p->out_layout;
  e->N = p->N;
  e->Cout = p->Cout;
  e->Do = pl.Do;
  e->Ho = pl.Ho;
  e->Wo = pl.Wo;
  e->flags = p->epi & ~static_cast<unsigned>(CONV3D_EPI_PAD_CACHE);
  e->bias = p->bias;
  e->residual = static_cast<const uint16_t*>(p->residual);
  e->rbias = p->residual_bias;
  e->gamma = p->gamma;
  e->value_out = static_cast<uint16_t*>(p->value_out);
  e->conv_out = static_cast<uint16_t*>(p->conv_out);
  e->sqrt_c = std::sqrt(static_cast<float>(p->Cout));
  e->halo = has_halo(p) ? 1 : 0;
  long long Dy, Hy, Wy;
  y_extent(p, pl.Do, pl.Ho, pl.Wo, &Dy, &Hy, &Wy);
  e->Dy = static_cast<int>(Dy);
  e->Hy = static_cast<int>(Hy);
  e->Wy = static_cast<int>(Wy);
  e->d0 = p->out_halo[0].before;
  e->h0 = p->out_halo[1].before;
  e->w0 = p->out_halo[2].before;
  e->h_mode = p->out_halo[1].mode == CONV3D_PAD_REFLECT ? 2 : 1;
  e->w_mode = p->out_halo[2].mode == CONV3D_PAD_REFLECT ? 2 : 1;
  e->up2 = p->input_upsample == 2 ? 1 : 0;
  e->acc_scale = 1.0f;
}

// Split of the reduction so that small layers still fill the GPU.  Each split
// adds work items (tiles x splits, run by persistent CTAs in waves of `sms`) and
// partial sums to reduce; the cost counted is waves x (stages per item + a fixed
// pipeline fill) + a small charge per split for the reduction pass.
int choose_splits(const conv3d_tuning& t, long long tiles, int stages_total, int sms, int* per) {
  int splits = t.k_splits;
  if (splits <= 0) {
    splits = 1;
    if (tiles < 2LL * sms) {
      double best = -1.0;
      const int smax = std::min(16, std::max(1, stages_total / 4));
      for (int s = 1; s <= smax; ++s) {
        const int p = static_cast<int>(cdiv(stages_total, s));
        const int se = static_cast<int>(cdiv(stages_total, p));
        if (se != s) continue;  // the same split as a smaller s
        const long long waves = cdiv(tiles * se, sms);
        const double cost = (double)waves * (p + 4) + (se > 1 ? 0.5 * se : 0.0);
        if (best < 0 || cost < best - 1e-9) {
          best = cost;
          splits = se;
        }
      }
    }
  }
  splits = std::max(1, std::min(splits, stages_total));
  *per = static_cast<int>(cdiv(stages_total, splits));
  return static_cast<int>(cdiv(stages_total, *per));
}

// Channel-major plan: M = 128 output channels, N = up to 256 output pixels.
int plan_cm(const conv3d_params* p, const conv3d_tuning& t, Plan* pl, size_t off) {
  ConvCMParams& k = pl->cp;
  std::memset(&k, 0, sizeof(k));
  const int Do = pl->Do, Ho = pl->Ho, Wo = pl->Wo;
  const int sw = p->stride[2];
  int kc = t.kc;
  if (kc == 0) kc = (pl->Cst > 32) ? 64 : (pl->Cst > 16 ? 32 : 16);
  if (kc != 16 && kc != 32 && kc != 64) return CONV3D_ERR_INVALID_ARG;
  k.kc = kc;
  k.row_bytes = kc * 2;
  k.n_chunks = static_cast<int>(cdiv(p->Cin, kc));
  // pixel tile
  bool halo, flat = false;
  int tw, rh;
  const bool flat_ok = sw == 1 && p->stride[1] == 1 && p->pad[2].before == 0 &&
                       p->pad[2].after == 0 &&
                       (p->pad[1].mode == CONV3D_PAD_ZERO ||
                        (p->pad[1].before == 0 && p->pad[1].after == 0));
  long long q_total = (long long)(Ho - 1) * p->W + Wo;  // flattened output range
  // flattened D*H*W: tiles run across frames, so small planes fill whole 256-pixel
  // tiles (no H / W padding: a row above the plane would be the previous frame's
  // last row; T zero padding reads positions outside the volume)
  const long long q3 = ((long long)(Do - 1) * p->H + (Ho - 1)) * p->W + Wo;
  const bool flat3_ok = flat_ok && p->stride[0] == 1 && p->pad[1].before == 0 &&
                        p->pad[1].after == 0 && p->pad[0].mode == CONV3D_PAD_ZERO &&
                        p->out_layout == CONV3D_NDHWC &&
                        !(p->epi & CONV3D_EPI_L2NORM_SILU) && t.kernel != 3 &&
                        q3 < 0x7fffff00LL;
  // Compact volume: the flattened volume without the KR - 1 input rows below each frame's
  // last output row (they hold no output position), walked by a TMA im2col map whose
  // bounding box spans W x Ho x Do.  Its corners (T: -pt and pad_after - (KT - 1), H:
  // 0 and -(KR - 1), W: 0 and 0) must lie in [-16, 15]; the im2col offsets (r, t) of a
  // copy stay within 0..2, the range measured on the hardware (KT, KR <= 3); every
  // channel chunk lies inside the tensor (the tiled maps zero-fill a partial last chunk).
  const long long qc = ((long long)(Do - 1) * Ho + (Ho - 1)) * p->W + Wo;
  const int up_t = p->pad[0].after - (p->KT - 1);
  const bool compact_ok = flat3_ok && t.compact != 2 && p->pad[0].before <= 16 &&
                          up_t >= -16 && up_t <= 15 && p->KT <= 3 && p->KR <= 3 &&
                          pl->Cst % kc == 0 && Ho == p->H - (p->KR - 1) && qc < 0x7fffff00LL;
  bool flat3 = false, compact = false;
  if (t.tile_w <= 0 && t.halo != 2 && flat_ok && q_total < 0x7fffff00LL) {
    // flattened H*W: a tile is 256 consecutive positions with row pitch W
    flat = true;
    halo = true;
    rh = 1;
    const long long tiles2 = (long long)Do * cdiv(q_total, std::min<long long>(256, round_up(q_total, 16)));
    const long long tiles3 = cdiv(q3, std::min<long long>(256, round_up(q3, 16)));
    const long long tilesc = cdiv(qc, std::min<long long>(256, round_up(qc, 16)));
    // Automatic only when it saves a round of tiles or 3 % of them, and not where the
    // paired last chunks would apply (the compact map has no half-width form).
    // (Ladder 256 -> 256 on [9, 64, 64] with a 1-pixel halo: 149 tiles against 153 per
    // channel tile, two rounds of 298 work items on 152 SMs instead of three; 512 ->
    // 512 on [5, 16, 16]: 6 against 7.)
    const long long best = std::min(tiles2, flat3_ok ? tiles3 : tiles2);
    const long long ct = cdiv(p->Cout, 128);
    const int sms_c = num_sms();
    const int last_c = pl->Cst - (k.n_chunks - 1) * kc;
    const bool pair_likely = t.pair != 2 && kc == 64 && last_c <= 32 && p->KT * p->KR >= 2;
    const bool compact_gain = tilesc < best && !pair_likely &&
                              (cdiv(tilesc * ct, sms_c) < cdiv(best * ct, sms_c) ||
                               tilesc * 100 <= best * 97);
    if (compact_ok && Do > 1 && (t.compact == 1 || compact_gain)) {
      flat3 = true;
      compact = true;
      q_total = qc;
    } else if (flat3_ok && Do > 1 && tiles3 < tiles2) {
      flat3 = true;
      q_total = q3;
    }
    tw = static_cast<int>(std::min<long long>(256, round_up(q_total, 16)));
    // Narrower tiles when the last wave of 256-wide tiles is nearly empty: a layer runs
    // in ceil(tiles / SMs) rounds of one tile per CTA, and a tile's time shrinks with
    // its width down to about 208 pixels (below that the per-stage latency sets it), so
    // the width with the fewest rounds x max(width, 208) wins when it saves at least 3 %.
    // Only for layers with at least a wave of tiles (smaller ones split the reduction).
    // (Ladder 256 -> 256 on [9, 64, 64]: 306 tiles = 2 waves + 2 tiles at width 256.)
    if (tw == 256) {
      const bool norm_units = (p->epi & CONV3D_EPI_L2NORM_SILU) != 0;
      const long long per_q = (flat3 ? 1LL : (long long)Do) * p->N *
                              (norm_units ? 1LL : cdiv(p->Cout, 128));
      const int sms0 = num_sms();
      auto cost = [&](int c) {
        const long long units = per_q * cdiv(q_total, c);
        return units < sms0 ? -1LL : cdiv(units, sms0) * std::max(c, 208);
      };
      const long long c256 = cost(256);
      if (c256 > 0) {
        long long best = c256;
        for (int c = 240; c >= 208; c -= 16) {
          const long long v = cost(c);
          if (v > 0 && v * 100 <= c256 * 97 && v < best) {
            best = v;
            tw = c;
          }
        }
      }
    }
  } else if (t.tile_w > 0) {
    tw = t.tile_w;
    rh = t.tile_h > 0 ? t.tile_h : 1;
    halo = (t.halo == 1) || (t.halo == 0 && sw == 1 && p->KS > 1 &&
                             rh * (tw + p->KS - 1) <= 256 + p->KS - 1);
  } else if (sw == 1 && p->KS > 1 && t.halo != 2) {
    // Strip tiles: rh output rows of tw pixels; each row's run of tw + KS - 1
    // input pixels sits run_pitch rows after the previous one, so one MMA of
    // N = (rh - 1) * pitch + tw rows covers the tile for every W tap.  The split
    // of the width (nt pieces) and of the rows is chosen to minimise MMA issue
    // time: an MMA costs about as much for N up to ~208 as for N = 208.
    long long best = -1;
    tw = 0;
    rh = 1;
    // NCDHW output: tile widths that are multiples of 8 keep every 32-pixel block of a row
    // on a column that is a multiple of 8, where the epilogue stores it with bulk tensor
    // stores (a block starting elsewhere takes the per-element path)
    const int wq = p->out_layout == CONV3D_NCDHW ? 8 : 1;
    for (int nt = 1; nt <= 16; ++nt) {
      const int ctw = static_cast<int>(round_up(cdiv(Wo, nt), wq));
      if (nt > 1 && (long long)(nt - 1) * ctw >= Wo) continue;  // a tile would be empty
      const int run = ctw + p->KS - 1;
      int crh, cN;
      if (run > 256) {
        if (ctw > 256) continue;
        crh = 1;
        cN = static_cast<int>(round_up(ctw, 16));
      } else {
        const int pitch = static_cast<int>(round_up(run, 8));  // runs stay 1024-byte aligned
        const int rmax = std::max(1, std::min((256 - ctw) / pitch + 1, Ho));
        const int nth = static_cast<int>(cdiv(Ho, rmax));
        crh = static_cast<int>(cdiv(Ho, nth));
        cN = static_cast<int>(round_up((long long)(crh - 1) * pitch + ctw, 16));
        if (cN > 256) continue;
      }
      const long long cost = (long long)std::max(cN, 208) * nt * cdiv(Ho, crh);
      if (best < 0 || cost < best) {
        best = cost;
        tw = ctw;
        rh = crh;
      }
    }
    if (best < 0) return CONV3D_ERR_UNSUPPORTED;
    // A layer that runs as one wave of work items (and too many items for a split of
    // its reduction) finishes with its slowest item: fewer rows per tile (a smaller N)
    // are faster as long as the items still fit in one wave.
    {
      const long long per_tile =
          (long long)Do * p->N * cdiv(p->Cout, 128) * (p->input_upsample == 2 ? 4 : 1);
      const int nt = static_cast<int>(cdiv(Wo, tw));
      const int pitch = static_cast<int>(round_up(tw + p->KS - 1, 8));
      auto items = [&](int r) { return nt * cdiv(Ho, r) * per_tile; };
      const int sms1 = num_sms();
      if (tw + p->KS - 1 <= 256 && items(rh) <= sms1 && 2 * items(rh) >= sms1) {
        while (rh > 1 && items(rh - 1) <= sms1 &&
               round_up((long long)(rh - 2) * pitch + tw, 16) <= 256)
          --rh;
      }
    }
    halo = true;
  } else {
    const int maxw = std::min(256, 256 / sw);
    tw = static_cast<int>(std::min<long long>(round_up(Wo, 8), maxw / 8 * 8));
    rh = std::max(1, std::min(256 / tw, Ho));
    halo = false;
  }
  if (halo && sw != 1) return CONV3D_ERR_INVALID_ARG;
  if (tw < 1 || rh < 1 || tw * sw > 256) return CONV3D_ERR_INVALID_ARG;
  k.tw = tw;
  k.rh = rh;
  k.halo = halo ? 1 : 0;
  k.flat = flat ? 1 : 0;
  k.flat3 = flat3 ? 1 : 0;
  k.compact = compact ? 1 : 0;
  k.tiles_d = flat3 ? 1 : Do;
  if (flat) {
    // (an im2col box takes up to 1024 pixels: one box a stage in the compact form)
    k.nbox = compact ? 1 : static_cast<int>(cdiv(tw + p->KS - 1, 256));
    k.box_w = k.nbox == 1 ? tw + p->KS - 1
                          : static_cast<int>(round_up(cdiv(tw + p->KS - 1, k.nbox), 8));
    k.run_pitch = k.nbox * k.box_w;
    k.N = static_cast<int>(round_up(tw, 16));
  } else if (halo) {
    const int run = tw + p->KS - 1;
    if (run > 256) {
      if (rh != 1) return CONV3D_ERR_INVALID_ARG;
      k.nbox = 2;
      k.box_w = static_cast<int>(round_up(cdiv(run, 2), 8));
    } else {
      k.nbox = 1;
      k.box_w = run;
    }
    // runs start on 8-row (swizzle-period) boundaries
    k.run_pitch = static_cast<int>(round_up((long long)k.nbox * k.box_w, 8));
    k.N = static_cast<int>(round_up((long long)(rh - 1) * k.run_pitch + tw, 16));
  } else {
    if (rh > 1 && tw % 8) return CONV3D_ERR_INVALID_ARG;
    k.nbox = 1;
    k.box_w = tw;
    k.run_pitch = tw;
    k.N = static_cast<int>(round_up((long long)tw * rh, 16));
    // the tile's rows are rh input rows sh apart: one copy with element stride sh along
    // H brings them all (the rows land tw apart, as the per-row copies place them),
    // unless a row needs the reflect-H coordinate mapping
    const bool reflect_h =
        p->pad[1].mode == CONV3D_PAD_REFLECT && (p->pad[1].before || p->pad[1].after);
    k.rows_box = (rh > 1 && !reflect_h && (long long)rh * p->stride[1] <= 256 &&
                  p->stride[1] <= 8) ? 1 : 0;
  }
  if (k.N > 256) return CONV3D_ERR_INVALID_ARG;
  // Pixel-major mode for layers with at most 128 output channels: N = Cout (rounded
  // to 16) over 128-pixel halves instead of M = 128 channel rows of which only Cout are
  // real; its epilogue (one pixel per thread) needs no staging.  Automatic for
  // Cout <= 16 (the RGB output convolution: 3 of 128 channel rows would be real);
  // measured slower than channel-major tiles on the 32- to 96-channel layers, where
  // it runs only on request (conv3d_tuning.kernel = 3).
  const bool up2 = p->input_upsample == 2;
  if (up2 && (!halo || flat || t.kernel == 3)) return CONV3D_ERR_UNSUPPORTED;
  const bool pm = !up2 && (t.kernel == 3 ||
                           (t.kernel == 0 && p->Cout <= 16 &&
                            !(p->epi & CONV3D_EPI_L2NORM_SILU) && !has_halo(p)));
  if (pm && p->Cout > 128) return CONV3D_ERR_UNSUPPORTED;
  k.pm = pm ? 1 : 0;
  if (pm) {
    k.N = static_cast<int>(round_up(k.N, 128));  // whole 128-pixel halves
    k.pm_halves = k.N / 128;
    k.pm_n = static_cast<int>(round_up(p->Cout, 16));
    k.pm_cols = static_cast<int>(round_up(k.pm_n, 32));
    k.wtap_rows = k.pm_n;
  } else {
    k.wtap_rows = 128;
  }
  k.taps_per_stage = halo ? p->KS : 1;
  k.stages_total = p->KT * p->KR * (halo ? 1 : p->KS) * k.n_chunks;
  const long long act_rows = std::max<long long>((long long)k.rh * k.run_pitch,
                                                 k.N + (halo ? p->KS - 1 : 0));
  k.act_bytes = static_cast<uint32_t>(round_up(round_up(act_rows, 8) * k.row_bytes, 1024));
  // Stages whose temporal tap reads only T padding are left out of a tile's range when
  // the tiles are long enough that the remaining stages still cover the epilogue of the
  // previous tile: on 9-stage tiles (e4m3 128->128) the short tiles of the first frames
  // were bound by epilogues (0.332 against 0.314 ms with every stage), on 18-stage tiles
  // (bf16 128->128) leaving them out gained (0.527 against 0.547 ms).
  k.skip_pad = (p->KT > 1 && k.stages_total >= 12 &&
                (p->pad[0].before > 0 || p->pad[0].after > 0)) ? 1 : 0;
  // Leading output frames whose first temporal taps read only the T padding have shorter
  // tiles (the kernel leaves those stages out).  With long tiles (36 stages or more, taps
  // folded into halo stages) they go last in the tile order, so that every CTA's last
  // round takes some of them: ladder 256->256 at [17, 128, 128] 0.525 -> 0.514 ms, at
  // [9, 64, 64] 0.105 -> 0.099 ms.  With shorter tiles the run of short tiles at the end
  // is bound by their epilogues and the plain order is faster (128->128: 0.518 against
  // 0.549 ms).  (Not for the paired schedule, which keeps every stage.)
  if (k.skip_pad && !flat3 && halo && p->pad[0].before > 0 && Do > 1 && k.stages_total >= 36) {
    const int dc = static_cast<int>(cdiv(p->pad[0].before, p->stride[0]));
    k.d_cheap = dc < Do ? dc : 0;
  }
  const uint32_t wgt_bytes = static_cast<uint32_t>(k.taps_per_stage * k.wtap_rows * k.row_bytes);
  k.stage_bytes = k.act_bytes + wgt_bytes;
  k.tiles_c = static_cast<int>(cdiv(p->Cout, 128));
  // fused L2 norm: den[N] in shared memory (channel-major; the pixel-major
  // epilogue owns whole channel rows)
  const bool norm = (p->epi & CONV3D_EPI_L2NORM_SILU) != 0 && !pm;
  const size_t norm_bytes = norm ? (size_t)k.N * 4 : 0;
  // Epilogue warpgroups: three hide the latency of the per-element work better
  // (layers with little reduction per output element are bound by it), two leave
  // room for one more pipeline stage.  Three unless that costs a stage on a layer
  // with a long reduction.
  auto stages_for = [&](int groups) {
    const size_t epi = pm ? 0 : (size_t)groups * 4 * kEpiWarpBytes;
    return static_cast<int>(std::min<size_t>(
        8, (kMaxSmem - 1024 - 256 - epi - norm_bytes) / k.stage_bytes));
  };
  const long long k_total = (long long)p->KT * p->KR * p->KS * p->Cin;
  const int epi_groups =
      pm ? 2 : ((stages_for(3) >= stages_for(2) || k_total <= 1152) ? 3 : 2);
  k.epi_groups = epi_groups;
  const size_t kEpiStage = pm ? 0 : (size_t)epi_groups * 4 * kEpiWarpBytes;
  int stages = stages_for(epi_groups);
  if (t.stages > 0) stages = std::min(stages, t.stages);
  if (stages < 2) return CONV3D_ERR_UNSUPPORTED;
  k.stages = stages;
  k.bar_off = k.stage_bytes * stages;
  // Only the rows of real output channels are loaded: out-of-bounds box rows
  // still cost transfer bandwidth.  The MMA reads all 128 rows; the rows past
  // Cout hold stale data and only reach accumulator lanes that are never stored.
  k.wgt_rows = static_cast<int>(std::min<long long>(128, round_up(p->Cout, 8)));
  k.wgt_rows_last = static_cast<int>(round_up(p->Cout - 128LL * (cdiv(p->Cout, 128) - 1), 8));
  {
    // Bytes one stage's copies deliver, counted the way the producer issues them:
    // per output row of the tile (one run for flat tiles) nbox boxes of box_w
    // pixels, then one weight box per tap.  A wrong count leaves the stage's
    // barrier incomplete or completes it early, so the plan is refused when the
    // closed form and the walk disagree.
    const int runs = flat ? 1 : k.rh;
    long long walked = 0;
    for (int i = 0; i < runs; ++i)
      for (int b = 0; b < k.nbox; ++b) walked += (long long)k.box_w * k.row_bytes;
    long long walked_last = walked;
    for (int tl = 0; tl < k.taps_per_stage; ++tl) {
      walked += (long long)k.wgt_rows * k.row_bytes;
      walked_last += (long long)k.wgt_rows_last * k.row_bytes;
    }
    const long long act_part = (long long)runs * k.nbox * k.box_w * k.row_bytes;
    const long long closed = act_part + (long long)k.taps_per_stage * k.wgt_rows * k.row_bytes;
    const long long closed_last =
        act_part + (long long)k.taps_per_stage * k.wgt_rows_last * k.row_bytes;
    if (walked != closed || walked_last != closed_last || closed >= (1LL << 20) ||
        closed_last >= (1LL << 20) || k.wgt_rows_last < 8 || k.wgt_rows_last > 128)
      return CONV3D_ERR_UNSUPPORTED;
    k.tx_bytes = static_cast<uint32_t>(closed);
    k.tx_bytes_last = static_cast<uint32_t>(closed_last);
    k.act_tx = static_cast<uint32_t>(act_part);
    // every loaded row must land inside the stage's activation / weight regions
    if ((long long)((runs - 1) * k.run_pitch + k.nbox * k.box_w) * k.row_bytes > k.act_bytes)
      return CONV3D_ERR_UNSUPPORTED;
  }
  k.tiles_w = static_cast<int>(flat ? cdiv(q_total, tw) : cdiv(Wo, tw));
  k.tiles_h = static_cast<int>(flat ? 1 : cdiv(Ho, rh));
  k.up2 = up2 ? 1 : 0;
  k.ncls = up2 ? 4 : 1;
  const long long tiles =
      (long long)k.tiles_w * k.tiles_h * k.tiles_d * p->N * k.tiles_c * k.ncls;
  const int sms = num_sms();
  int per = 0;
  // with the fused norm the channel tiles of a pixel tile share a CTA, so the
  // parallelism that decides the split is the number of pixel tiles
  const long long par = norm ? tiles / k.tiles_c : tiles;
  // Paired last chunks: the last 64-channel chunk of a tap pair holds at most 32 real
  // channels, so two tap pairs share one stage of 32-channel rows (every stage then
  // carries a full 64-channel MMA group).  One split only; not with the reflect-W
  // patch (it rewrites 128-byte rows) or the pixel-major mode.  From two tap pairs up
  // (3x3x3: 18 -> 14 stages for 96 channels; 1x3x3: 6 -> 5; both about -5 % time
  // measured once every stage issues its MMAs from straight-line code).
  const int n_pairs = p->KT * p->KR;
  const int last_ch = pl->Cst - (k.n_chunks - 1) * kc;
  const bool reflect_w_pad =
      p->pad[2].mode == CONV3D_PAD_REFLECT && (p->pad[2].before || p->pad[2].after);
  const bool pair_ok = t.pair != 2 && !pm && !up2 && !compact && halo && kc == 64 &&
                       last_ch >= 1 && last_ch <= 32 && n_pairs >= 2 && !reflect_w_pad;
  int splits = 0;
  if (pair_ok) {
    const int total = n_pairs * (k.n_chunks - 1) + (n_pairs + 1) / 2;
    splits = choose_splits(t, par, total, sms, &per);
    if (splits == 1) {
      k.pair = 1;
      k.d_cheap = 0;  // every stage of the paired schedule runs
      k.skip_pad = 0;
      k.stages_total = total;
    }
  }
  if (!k.pair) {
    conv3d_tuning t1 = t;
    if (up2) t1.k_splits = 1;  // the split reduction writes plain output pixels
    splits = choose_splits(t1, par, k.stages_total, sms, &per);
  }
  k.n_pairs = n_pairs;
  k.k_splits = splits;
  k.stages_per_split = per;
  if (tiles * splits > 0x7fffffffLL) return CONV3D_ERR_UNSUPPORTED;
  k.num_tiles = static_cast<int>(tiles * splits);
  k.norm = (norm && splits == 1) ? 1 : 0;
  k.tpu = k.norm ? k.tiles_c : 1;
  // bulk tensor stores for the output blocks that lie on one output row: NDHWC,
  // value = B(B(conv) + bias) (no residual, norm or bottom/right pad), 16-byte rows
  // (NCDHW: 16-byte output rows, and no NDHWC debug conv store beside them)
  const bool store_rows = p->out_layout == CONV3D_NDHWC
                              ? p->Cout % 8 == 0
                              : (Wo % 8 == 0 && !(p->epi & CONV3D_EPI_DEBUG_STORE_CONV));
  k.tma_store = (store_rows && splits == 1 && !pm &&
                 !(p->epi & (CONV3D_EPI_RESIDUAL | CONV3D_EPI_L2NORM_SILU |
                             CONV3D_EPI_OUT_PAD_BR)) &&
                 !(up2 && (p->epi & CONV3D_EPI_DEBUG_STORE_CONV)))
                    ? 1
                    : 0;
  k.acc_cols = pm ? k.pm_halves * k.pm_cols : static_cast<int>(round_up(k.N, 32));
  k.nbuf = (2 * k.acc_cols <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < k.nbuf * k.acc_cols) cols *= 2;
  k.tmem_cols = cols;
  k.M_total = (long long)p->N * Do * Ho * Wo;
  if (splits > 1) {
    pl->partial_off = off;
    pl->partial_bytes = (size_t)splits * (size_t)k.M_total * p->Cout * 4;
    off = static_cast<size_t>(round_up(off + pl->partial_bytes, 256));
  }
  const int grid = static_cast<int>(std::min<long long>(k.num_tiles / k.tpu, sms));
  // Weight L2 prefetch: when each CTA runs at most a few work items, every weight
  // slice it loads is a first read from HBM (the slices of one channel tile and split
  // are shared by few pixel tiles), and the two-stage pipeline waits for it; asking L2
  // for the weights some stages ahead overlaps those reads.  Layers whose CTAs loop
  // over many tiles find the weights in L2 already.
  // (Measured on the ladder's 16x16 layers: 512->512 -4 %, 1024->1024 -9 % at 4 stages
  // ahead; layers with a few MB of weights gained nothing, so they stay off.)
  const size_t wbytes = (size_t)p->Cout * p->KT * p->KR * p->KS * round_up(p->Cin, 64) * 2;
  if (t.prefetch > 0)
    k.wpref = t.prefetch;
  else if (t.prefetch == 0 && !k.pair && k.num_tiles <= 4LL * grid && wbytes >= (8u << 20))
    k.wpref = 4;
  else
    k.wpref = 0;
  if (k.norm) {
    k.norm_cs = static_cast<int>(round_up(p->Cout, 8));
    pl->vscratch_off = off;
    pl->vscratch_bytes = (size_t)grid * k.N * k.norm_cs * 2;
    off = static_cast<size_t>(round_up(off + pl->vscratch_bytes, 256));
  }
  pl->ws_bytes = off;
  pl->grid = dim3(static_cast<unsigned>(grid), 1, 1);
  k.epi_off = k.bar_off + 256;
  k.norm_off = static_cast<uint32_t>(k.epi_off + kEpiStage);
  pl->smem = 1024 + k.norm_off + norm_bytes;
  pl->launches = (pl->stage ? 1 : 0) + 1 + (splits > 1 ? 1 : 0);
  k.C = pl->Cst;
  k.D = p->D;
  k.H = p->H;
  k.W = p->W;
  k.KT = p->KT;
  k.KR = p->KR;
  k.KS = p->KS;
  k.st = p->stride[0];
  k.sh = p->stride[1];
  k.sw = sw;
  k.pt = p->pad[0].before;
  k.ph = p->pad[1].before;
  k.pw = p->pad[2].before;
  k.reflect_h = (p->pad[1].mode == CONV3D_PAD_REFLECT && (p->pad[1].before || p->pad[1].after));
  k.reflect_w = (p->pad[2].mode == CONV3D_PAD_REFLECT && (p->pad[2].before || p->pad[2].after));
  k.cp64 = static_cast<int>(round_up(p->Cin, 64));
  k.inject = t.inject;
  k.timeout_ns = (unsigned long long)(t.timeout_ms > 0 ? t.timeout_ms : default_timeout_ms()) *
                 1000000ULL;
  fill_epi(p, *pl, &k.epi);
  return CONV3D_OK;
}

// Narrow-input gather plan (Cin < 8, KR * KS * Cin <= 32, stride 1 along W, W
// padding <= 1): channel-major tiles of one output row (N = up to 256 pixels), one
// stage per temporal tap whose K = KR * KS * Cin values are gathered in shared
// memory from TMA copies of the raw input rows (ConvCMParams::gather); no staged
// copy of the input and no separate launch.  Returns CONV3D_ERR_UNSUPPORTED when
// the shape does not fit it.
int plan_gather(const conv3d_params* p, const conv3d_tuning& t, Plan* pl) {
  ConvCMParams& k = pl->cp;
  std::memset(&k, 0, sizeof(k));
  const int Do = pl->Do, Ho = pl->Ho, Wo = pl->Wo;
  const int C = p->Cin;
  const bool cl = p->layout == CONV3D_NDHWC;
  const int krs = p->KR * p->KS;
  const bool pads_ok = p->pad[2].before <= 1 && p->pad[2].after <= 1 &&
                       (p->pad[1].mode == CONV3D_PAD_ZERO ||
                        (p->pad[1].before <= 1 && p->pad[1].after <= 1));
  if (C >= 8 || krs < 2 || krs * C > 32 || p->stride[2] != 1 || !pads_ok ||
      (p->epi & CONV3D_EPI_L2NORM_SILU) || (cl ? ((long long)p->W * C) % 8 : p->W % 8) != 0)
    return CONV3D_ERR_UNSUPPORTED;
  const int tiles_c = static_cast<int>(cdiv(p->Cout, 128));
  const size_t wres_bytes = (size_t)tiles_c * p->KT * 128 * 64;
  if (wres_bytes > (64u << 10)) return CONV3D_ERR_UNSUPPORTED;
  k.gather = 1;
  k.kc = 32;
  k.row_bytes = 64;
  k.n_chunks = 1;
  k.tw = std::min(Wo, 256);
  k.rh = 1;
  k.halo = 0;
  k.nbox = 1;
  k.box_w = k.tw;
  k.run_pitch = k.tw;
  k.N = static_cast<int>(round_up(k.tw, 16));
  k.wtap_rows = 128;
  k.taps_per_stage = 1;
  k.stages_total = p->KT;
  k.g_K = krs * C;
  k.g_cpp = cl ? C : 1;
  k.g_planes = cl ? 1 : C;
  // groups of 8 values per raw row: the row's first group is rounded down, so one
  // more group than the values cover; rows are whole 128-byte lines
  const long long vals = (long long)(k.tw + p->KS - 1) * k.g_cpp;
  const int nG = static_cast<int>(round_up(cdiv(vals + 7, 8), 8));
  if (nG > 256) return CONV3D_ERR_UNSUPPORTED;
  k.g_row_bytes = nG * 16;
  const int raw_rows = k.g_planes * p->KR;
  k.g_raw_off = static_cast<uint32_t>(round_up((long long)k.N * 64, 1024));
  k.act_bytes = k.g_raw_off;
  k.stage_bytes = static_cast<uint32_t>(
      round_up(k.g_raw_off + (long long)raw_rows * k.g_row_bytes, 1024));
  k.tx_bytes = k.tx_bytes_last = k.act_tx = static_cast<uint32_t>(raw_rows * k.g_row_bytes);
  k.wgt_rows = static_cast<int>(std::min<long long>(128, round_up(p->Cout, 8)));
  k.wgt_rows_last = static_cast<int>(round_up(p->Cout - 128LL * (tiles_c - 1), 8));
  k.tiles_c = tiles_c;
  auto stages_for = [&](int groups) {
    const size_t epi = (size_t)groups * 4 * kEpiWarpBytes;
    const long long avail = (long long)kMaxSmem - 1024 - 256 - (long long)epi -
                            (long long)wres_bytes - 1024;
    return static_cast<int>(std::min<long long>(8, std::max<long long>(0, avail / k.stage_bytes)));
  };
  const int epi_groups = 3;
  k.epi_groups = epi_groups;
  int stages = stages_for(epi_groups);
  if (t.stages > 0) stages = std::min(stages, t.stages);
  if (stages < 2) return CONV3D_ERR_UNSUPPORTED;
  k.stages = stages;
  k.bar_off = k.stage_bytes * stages;
  k.tiles_w = static_cast<int>(cdiv(Wo, k.tw));
  k.tiles_h = Ho;
  k.tiles_d = Do;
  const long long tiles = (long long)k.tiles_w * Ho * Do * p->N * tiles_c;
  if (tiles > 0x7fffffffLL) return CONV3D_ERR_UNSUPPORTED;
  k.k_splits = 1;
  k.stages_per_split = p->KT;
  k.num_tiles = static_cast<int>(tiles);
  k.tpu = 1;
  const bool store_rows = p->out_layout == CONV3D_NDHWC
                              ? p->Cout % 8 == 0
                              : (Wo % 8 == 0 && !(p->epi & CONV3D_EPI_DEBUG_STORE_CONV));
  k.tma_store = (store_rows && !(p->epi & (CONV3D_EPI_RESIDUAL | CONV3D_EPI_OUT_PAD_BR))) ? 1 : 0;
  k.acc_cols = static_cast<int>(round_up(k.N, 32));
  k.nbuf = (2 * k.acc_cols <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < k.nbuf * k.acc_cols) cols *= 2;
  k.tmem_cols = cols;
  k.M_total = (long long)p->N * Do * Ho * Wo;
  const int sms = num_sms();
  const int grid = static_cast<int>(std::min<long long>(k.num_tiles, sms));
  pl->ws_bytes = 0;
  pl->grid = dim3(static_cast<unsigned>(grid), 1, 1);
  k.epi_off = k.bar_off + 256;
  k.norm_off = static_cast<uint32_t>(k.epi_off + (size_t)epi_groups * 4 * kEpiWarpBytes);
  k.g_wres_off = static_cast<uint32_t>(round_up(k.norm_off, 1024));
  pl->smem = 1024 + k.g_wres_off + wres_bytes;
  if (pl->smem > kMaxSmem) return CONV3D_ERR_UNSUPPORTED;
  pl->launches = 1;
  pl->stage = false;
  pl->Cst = C;
  k.C = C;
  k.D = p->D;
  k.H = p->H;
  k.W = p->W;
  k.KT = p->KT;
  k.KR = p->KR;
  k.KS = p->KS;
  k.st = p->stride[0];
  k.sh = p->stride[1];
  k.sw = 1;
  k.pt = p->pad[0].before;
  k.ph = p->pad[1].before;
  k.pw = p->pad[2].before;
  k.reflect_h = (p->pad[1].mode == CONV3D_PAD_REFLECT && (p->pad[1].before || p->pad[1].after));
  k.reflect_w = (p->pad[2].mode == CONV3D_PAD_REFLECT && (p->pad[2].before || p->pad[2].after));
  k.cp64 = static_cast<int>(round_up(p->Cin, 64));
  k.inject = t.inject;
  k.timeout_ns = (unsigned long long)(t.timeout_ms > 0 ? t.timeout_ms : default_timeout_ms()) *
                 1000000ULL;
  fill_epi(p, *pl, &k.epi);
  return CONV3D_OK;
}

// Pixel-major plan: M = 128 output pixels per tile, N = output channels (a tile
// holds a pixel's whole channel row).  Used when no channel-major plan fits, or
// on request (conv3d_tuning.kernel = 1).
int plan_pm(const conv3d_params* p, const conv3d_tuning& t, Plan* pl, size_t off) {
  const int Do = pl->Do, Ho = pl->Ho, Wo = pl->Wo;
  const int st = p->stride[0], sh = p->stride[1], sw = p->stride[2];
  const bool norm = (p->epi & CONV3D_EPI_L2NORM_SILU) != 0;
  ConvTCParams& k = pl->kp;
  std::memset(&k, 0, sizeof(k));
  // ---- channel chunk ----
  int kc = t.kc;
  if (kc == 0) kc = (pl->Cst % 64 == 0) ? 64 : (pl->Cst % 32 == 0) ? 32 : 16;
  if (kc != 16 && kc != 32 && kc != 64) return CONV3D_ERR_INVALID_ARG;
  k.kc = kc;
  k.row_bytes = kc * 2;
  k.swz = (kc == 64) ? 2 : (kc == 32) ? 4 : 6;
  k.n_chunks = static_cast<int>(cdiv(p->Cin, kc));

  // ---- N tiling ----
  int BN, n_sub, sub_n;
  if (norm) {
    BN = static_cast<int>(round_up(p->Cout, 16));
    n_sub = static_cast<int>(cdiv(BN, 256));
    sub_n = static_cast<int>(round_up(cdiv(BN, n_sub), 16));
    BN = n_sub * sub_n;
    if (BN > 512) return CONV3D_ERR_UNSUPPORTED;
  } else if (t.BN > 0) {
    if (t.BN % 16 || t.BN > 256) return CONV3D_ERR_INVALID_ARG;
    BN = t.BN;
    n_sub = 1;
    sub_n = BN;
  } else {
    const int nt = static_cast<int>(cdiv(p->Cout, 256));
    BN = static_cast<int>(round_up(cdiv(p->Cout, nt), 16));
    n_sub = 1;
    sub_n = BN;
  }
  const int n_tiles = static_cast<int>(cdiv(p->Cout, BN));
  k.BN = BN;
  k.n_sub = n_sub;
  k.sub_n = sub_n;
  k.acc_stride = static_cast<int>(round_up(BN, 32));

  // ---- M tile ----
  int tile_w = t.tile_w, tile_h = t.tile_h;
  if (tile_w <= 0) {
    if (Wo >= 128) {
      tile_w = 128;
      tile_h = 1;
    } else {
      tile_w = static_cast<int>(round_up(Wo, 8));
      if (tile_h <= 0) tile_h = std::max(1, std::min(128 / tile_w, Ho));
    }
  }
  if (tile_h <= 0) tile_h = 1;
  while (tile_w * sw > 256) tile_w -= 8;
  if (tile_w < 1 || tile_w > 128 || tile_w * tile_h > 128) return CONV3D_ERR_INVALID_ARG;
  if (tile_h > 1 && tile_w % 8) return CONV3D_ERR_INVALID_ARG;
  bool halo = (sw == 1 && tile_h == 1 && p->KS > 1);
  if (t.halo == 2) halo = false;
  if (t.halo == 1) {
    if (sw != 1 || tile_h != 1) return CONV3D_ERR_INVALID_ARG;
    halo = true;
  }
  k.tile_w = tile_w;
  k.tile_h = tile_h;
  k.halo = halo ? 1 : 0;
  k.box_w = halo ? tile_w + p->KS - 1 : tile_w;
  k.pitch_rows = static_cast<int>(round_up(k.box_w, 8));
  if (tile_h > 1) k.pitch_rows = tile_w;  // rows of one M-tile must be contiguous
  k.a_tile_rows = tile_h * k.pitch_rows;
  k.taps_per_stage = halo ? p->KS : 1;
  k.stages_total = p->KT * p->KR * (halo ? 1 : p->KS) * k.n_chunks;

  const int tiles_w = static_cast<int>(cdiv(Wo, tile_w));
  const int sms = num_sms();
  // ---- R (M-tiles per CTA) and pipeline depth ----
  int Rmax = std::max(1, std::min(4, 512 / k.acc_stride));
  if (t.R > 0) Rmax = t.R;
  int R = Rmax;
  size_t a_stage = 0, b_stage = 0;
  int stages = 0;
  for (; R >= 1; --R) {
    if (R * k.acc_stride > 512) continue;
    const long long groups_h = cdiv(Ho, (long long)R * tile_h);
    const long long ctas = (long long)tiles_w * groups_h * Do * p->N * n_tiles;
    if (t.R == 0 && R > 1 && ctas < 2LL * sms) continue;
    const long long a_rows = (long long)(R - 1) * k.a_tile_rows +
                             std::max<long long>(k.a_tile_rows, 128 + (halo ? p->KS - 1 : 0));
    a_stage = static_cast<size_t>(round_up(round_up(a_rows, 8) * k.row_bytes, 1024));
    b_stage = static_cast<size_t>(round_up((long long)k.taps_per_stage * BN * k.row_bytes, 1024));
    const size_t avail = kMaxSmem - 1024 - 256;
    stages = static_cast<int>(std::min<size_t>(8, avail / (a_stage + b_stage)));
    if (t.stages > 0) stages = std::min(stages, t.stages);
    if (stages >= 2) break;
    if (R == 1 && halo && t.halo != 1) {
      // the KS weight boxes of a halo stage do not fit twice: load one tap per stage
      halo = false;
      k.halo = 0;
      k.box_w = tile_w;
      k.pitch_rows = static_cast<int>(round_up(k.box_w, 8));
      if (tile_h > 1) k.pitch_rows = tile_w;
      k.a_tile_rows = tile_h * k.pitch_rows;
      k.taps_per_stage = 1;
      k.stages_total = p->KT * p->KR * p->KS * k.n_chunks;
      R = Rmax + 1;  // retry every R without the halo
    }
  }
  if (R < 1 || stages < 2) return CONV3D_ERR_UNSUPPORTED;
  k.R = R;
  k.stages = stages;
  k.a_stage_bytes = static_cast<uint32_t>(a_stage);
  k.b_stage_bytes = static_cast<uint32_t>(b_stage);
  k.bar_off = static_cast<uint32_t>((a_stage + b_stage) * stages);
  int cols = 32;
  while (cols < R * k.acc_stride) cols *= 2;
  k.tmem_cols = cols;
  k.tiles_w = tiles_w;
  k.groups_h = static_cast<int>(cdiv(Ho, (long long)R * tile_h));
  k.tx_bytes = static_cast<uint32_t>((long long)R * tile_h * k.box_w * k.row_bytes +
                                     (long long)k.taps_per_stage * n_sub * sub_n * k.row_bytes);

  // ---- split of the reduction ----
  const long long m_groups = (long long)tiles_w * k.groups_h * Do * p->N;
  const long long ctas = m_groups * n_tiles;
  int splits = t.k_splits;
  if (splits <= 0) {
    splits = 1;
    if (ctas < sms) {
      splits = static_cast<int>(std::max<long long>(1, (sms + ctas / 2) / ctas));
      splits = std::min(splits, std::max(1, k.stages_total / 4));
      splits = std::min(splits, 16);
    }
  }
  splits = std::max(1, std::min(splits, k.stages_total));
  int per = static_cast<int>(cdiv(k.stages_total, splits));
  splits = static_cast<int>(cdiv(k.stages_total, per));
  k.k_splits = splits;
  k.stages_per_split = per;
  k.M_total = (long long)p->N * Do * Ho * Wo;
  if (splits > 1) {
    pl->partial_off = off;
    pl->partial_bytes = (size_t)splits * (size_t)k.M_total * p->Cout * 4;
    off = static_cast<size_t>(round_up(off + pl->partial_bytes, 256));
  }
  pl->ws_bytes = off;
  if (m_groups > 0x7fffffffLL || n_tiles > 65535 || splits > 65535) return CONV3D_ERR_UNSUPPORTED;
  pl->grid = dim3(static_cast<unsigned>(m_groups), static_cast<unsigned>(n_tiles),
                  static_cast<unsigned>(splits));
  pl->smem = 1024 + k.bar_off + 8 * (3 * stages + 2) + 16;
  pl->launches = (pl->stage ? 1 : 0) + 1 + (splits > 1 ? 1 : 0);

  // ---- geometry ----
  k.C = pl->Cst;
  k.D = p->D;
  k.H = p->H;
  k.W = p->W;
  k.KT = p->KT;
  k.KR = p->KR;
  k.KS = p->KS;
  k.st = st;
  k.sh = sh;
  k.sw = sw;
  k.pt = p->pad[0].before;
  k.ph = p->pad[1].before;
  k.pw = p->pad[2].before;
  k.reflect_h = (p->pad[1].mode == CONV3D_PAD_REFLECT && (p->pad[1].before || p->pad[1].after));
  k.reflect_w = (p->pad[2].mode == CONV3D_PAD_REFLECT && (p->pad[2].before || p->pad[2].after));
  k.cp64 = static_cast<int>(round_up(p->Cin, 64));
  k.inject = t.inject;
  k.timeout_ns = (unsigned long long)(t.timeout_ms > 0 ? t.timeout_ms : default_timeout_ms()) *
                 1000000ULL;

  fill_epi(p, *pl, &k.epi);
  return CONV3D_OK;
}

int make_plan_conv(const conv3d_params* p, const conv3d_tuning* tu, Plan* pl) {
  int rc = validate_shape(p, &pl->Do, &pl->Ho, &pl->Wo);
  if (rc) return rc;
  rc = check_supported(p);
  if (rc) return rc;
  conv3d_tuning t{};
  if (tu) t = *tu;
  if (p->dtype == CONV3D_DTYPE_E4M3) {
    // e4m3 operands: a K step of the f8f6f4 MMA (32 one-byte channels) spans the same
    // 32 bytes as a bf16 K step, so the channel-major plan of the same convolution over
    // Cin / 2 two-byte channel pairs describes every copy and shared-memory layout;
    // only the MMA kind and the accumulator scale differ
    if (t.kernel == 1 || t.kernel == 3 || t.im2col == 1 || t.im2col == 3)
      return CONV3D_ERR_UNSUPPORTED;
    conv3d_params q = *p;
    q.Cin = p->Cin / 2;
    q.dtype = CONV3D_DTYPE_BF16;
    conv3d_tuning t2 = t;
    t2.pair = 2;  // one plain schedule for the e4m3 instances
    pl->f8 = true;
    pl->cm = true;
    pl->Cst = q.Cin;
    pl->q = q;
    rc = plan_cm(&pl->q, t2, pl, 0);
    if (rc) return rc;
    if (pl->cp.pm || pl->cp.gather || pl->cp.up2 || pl->cp.pair) return CONV3D_ERR_UNSUPPORTED;
    pl->cp.f8 = 1;
    pl->cp.epi.acc_scale = p->fp8_scale;
    return CONV3D_OK;
  }
  if (p->input_upsample == 2) {
    // x2 upsampled input: the channel-major kernel tiles the low-resolution grid (a
    // 3x3, pad-1 convolution of it, once per parity class); the output is twice as
    // large along H and W
    if (t.kernel == 1 || t.kernel == 3) return CONV3D_ERR_UNSUPPORTED;
    pl->stage = (p->layout == CONV3D_NCDHW) || (p->Cin % 8 != 0);
    pl->Cst = static_cast<int>(round_up(p->Cin, 8));
    size_t off0 = 0;
    if (pl->stage) {
      pl->stage_off = 0;
      pl->stage_bytes = (size_t)p->N * p->D * p->H * p->W * pl->Cst * 2;
      off0 = static_cast<size_t>(round_up(pl->stage_bytes, 256));
    }
    const int Ho = pl->Ho, Wo = pl->Wo;
    pl->Ho = p->H;
    pl->Wo = p->W;
    pl->cm = true;
    rc = plan_cm(p, t, pl, off0);
    pl->Ho = Ho;
    pl->Wo = Wo;
    return rc;
  }
  size_t off = 0;
  const int krs = p->KR * p->KS;
  // Narrow input: gather the taps in the convolution kernel itself.  Automatic for
  // one temporal tap (the T = 1 image layers: 3->96 at 1024^2 0.128 -> 0.105 ms);
  // with KT > 1 every input row is expanded once per temporal tap, and the staged
  // gather below, which expands each row once, measured faster (conv_in 3->128 on
  // [17, 256, 256]: 0.151 ms staged, 0.189 ms in the kernel).
  if ((t.im2col == 3 || (t.im2col == 0 && p->KT == 1)) && t.kernel != 1) {
    const Plan before = *pl;
    pl->cm = true;
    rc = plan_gather(p, t, pl);
    if (rc == CONV3D_OK || t.im2col == 3) return rc;
    *pl = before;
  }
  if (t.im2col != 2 && krs > 1 && p->Cin < 8 && (long long)krs * p->Cin <= 64 &&
      pl->Ho <= 65535 && (long long)p->N * p->D <= 65535) {
    // narrow input: gather the KR x KS spatial taps of every output pixel
    pl->im2col = true;
    pl->stage = true;
    pl->Ck = static_cast<int>(round_up((long long)krs * p->Cin, 16));
    pl->Cst = pl->Ck;
    pl->stage_off = 0;
    pl->stage_bytes = (size_t)p->N * p->D * pl->Ho * pl->Wo * pl->Ck * 2;
    off = static_cast<size_t>(round_up(pl->stage_bytes, 256));
    pl->wr_off = off;
    pl->wr_bytes = (size_t)p->Cout * p->KT * round_up(pl->Ck, 64) * 2;
    off = static_cast<size_t>(round_up(off + pl->wr_bytes, 256));
    conv3d_params q = *p;
    q.layout = CONV3D_NDHWC;
    q.Cin = pl->Ck;
    q.H = pl->Ho;
    q.W = pl->Wo;
    q.KR = q.KS = 1;
    q.stride[1] = q.stride[2] = 1;
    for (int i = 1; i < 3; ++i) {
      q.pad[i].before = q.pad[i].after = 0;
      q.pad[i].mode = CONV3D_PAD_ZERO;
    }
    pl->q = q;
    if (t.kernel == 1) {
      pl->cm = false;
      return plan_pm(&pl->q, t, pl, off);
    }
    pl->cm = true;
    return plan_cm(&pl->q, t, pl, off);
  }
  // input staging: NCDHW input, or channels not a multiple of 8 (TMA strides)
  pl->stage = (p->layout == CONV3D_NCDHW) || (p->Cin % 8 != 0);
  pl->Cst = static_cast<int>(round_up(p->Cin, 8));
  if (pl->stage) {
    pl->stage_off = off;
    pl->stage_bytes = (size_t)p->N * p->D * p->H * p->W * pl->Cst * 2;
    off = static_cast<size_t>(round_up(off + pl->stage_bytes, 256));
  }
  if (t.kernel == 1) {
    pl->cm = false;
    return plan_pm(p, t, pl, off);
  }
  const Plan before = *pl;
  pl->cm = true;
  rc = plan_cm(p, t, pl, off);
  if (rc != CONV3D_ERR_UNSUPPORTED || t.kernel == 2 || t.kernel == 3) return rc;
  // no channel-major plan for this shape: pixel-major tiles
  *pl = before;
  pl->cm = false;
  return plan_pm(p, t, pl, off);
}

int check_pointers(const conv3d_params* p, const Plan& pl) {
  auto mis = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u); };
  if (mis(p->x) || mis(p->w_packed) || mis(p->y) || mis(p->residual) || mis(p->value_out) ||
      mis(p->conv_out) || mis(p->bias) || mis(p->residual_bias) || mis(p->gamma) ||
      (pl.ws_bytes && mis(p->workspace)) || (pl.pad_cache && mis(p->cache_out)))
    return CONV3D_ERR_MISALIGNED;
  if (pl.ws_bytes && (!p->workspace || p->workspace_bytes < pl.ws_bytes))
    return CONV3D_ERR_WORKSPACE;
  const bool padbr = (p->epi & CONV3D_EPI_OUT_PAD_BR) != 0;
  const size_t out_elems = (size_t)p->N * p->Cout * pl.Do * pl.Ho * pl.Wo;
  long long Dy, Hy, Wy;
  y_extent(p, pl.Do, pl.Ho, pl.Wo, &Dy, &Hy, &Wy);
  const size_t y_elems =
      pl.pad_cache
          ? (size_t)p->N * p->Cout * (pl.Do + 2) * (pl.Ho + 2) * (pl.Wo + 2)
          : (size_t)p->N * p->Cout * Dy * (Hy + (padbr ? 1 : 0)) * (Wy + (padbr ? 1 : 0));
  const size_t cache_elems = pl.pad_cache ? (size_t)p->N * p->Cout * pl.Ho * pl.Wo *
                                                std::min(2, pl.Do + p->history_frames)
                                          : 0;
  auto span = [](const void* q, size_t bytes) {
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(q);
    s.hi = q ? s.lo + bytes : s.lo;
    return s;
  };
  const bool f8 = p->dtype == CONV3D_DTYPE_E4M3;
  const Span in[] = {
      span(p->x, (size_t)p->N * p->Cin * p->D * p->H * p->W * (f8 ? 1 : 2)),
      span(p->w_packed, f8 ? conv3d_packed_weight_bytes_e4m3(p->Cout, p->Cin, p->KT, p->KR, p->KS)
                           : conv3d_packed_weight_bytes(p->Cout, p->Cin, p->KT, p->KR, p->KS)),
      span((p->epi & CONV3D_EPI_RESIDUAL) ? p->residual : nullptr, out_elems * 2),
      span((p->epi & CONV3D_EPI_BIAS) ? p->bias : nullptr, (size_t)p->Cout * 4),
      span((p->epi & CONV3D_EPI_RESIDUAL_BIAS) ? p->residual_bias : nullptr, (size_t)p->Cout * 4),
      span((p->epi & CONV3D_EPI_L2NORM_SILU) ? p->gamma : nullptr, (size_t)p->Cout * 4),
  };
  const Span out[] = {
      span(p->y, y_elems * 2),
      span((p->epi & CONV3D_EPI_SAVE_VALUE) ? p->value_out : nullptr, out_elems * 2),
      span((p->epi & CONV3D_EPI_DEBUG_STORE_CONV) ? p->conv_out : nullptr, out_elems * 2),
      span(pl.ws_bytes ? p->workspace : nullptr, pl.ws_bytes),
      span(pl.pad_cache ? p->cache_out : nullptr, cache_elems * 2),
  };
  for (size_t i = 0; i < sizeof(out) / sizeof(out[0]); ++i) {
    for (size_t j = 0; j < sizeof(in) / sizeof(in[0]); ++j)
      if (overlaps(out[i], in[j])) return CONV3D_ERR_OVERLAP;
    for (size_t j = i + 1; j < sizeof(out) / sizeof(out[0]); ++j)
      if (overlaps(out[i], out[j])) return CONV3D_ERR_OVERLAP;
  }
  return CONV3D_OK;
}

// The plan of a call: the convolution's own plan, plus (padded output + cache) the
// scratch activation buffer after its workspace and the launch that places them.
int make_plan(const conv3d_params* p, const conv3d_tuning* tu, Plan* pl) {
  const int rc = make_plan_conv(p, tu, pl);
  if (rc || !(p->epi & CONV3D_EPI_PAD_CACHE)) return rc;
  pl->pad_cache = true;
  pl->pc_off = static_cast<size_t>(round_up(pl->ws_bytes, 256));
  pl->pc_bytes = (size_t)p->N * pl->Do * pl->Ho * pl->Wo * p->Cout * 2;
  pl->ws_bytes = pl->pc_off + pl->pc_bytes;
  pl->launches += 1;
  return CONV3D_OK;
}

// ---- TMA descriptors ----------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

using EncodeIm2colFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const int*, const int*,
                                    cuuint32_t, cuuint32_t, const cuuint32_t*,
                                    CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeIm2colFn encode_im2col_fn() {
  static EncodeIm2colFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeIm2colFn>(ptr);
  }
  return fn;
}

CUtensorMapSwizzle swizzle_of(int kc) {
  return kc == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                  : (kc == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

int encode_maps(const conv3d_params* p, const Plan& pl, const void* xin, CUtensorMap* tmA,
                CUtensorMap* tmB, CUtensorMap* tmBLast, vvc::CmHalfMaps* half) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return CONV3D_ERR_CUDA;
  int kc, act_box, es_w, wgt_rows, wgt_rows_last, cp64;
  bool flat = false;
  if (pl.cm) {
    const ConvCMParams& k = pl.cp;
    flat = k.flat != 0;
    kc = k.kc;
    act_box = k.halo ? k.box_w : k.box_w * k.sw;
    es_w = k.halo ? 1 : k.sw;
    wgt_rows = k.wgt_rows;
    wgt_rows_last = k.wgt_rows_last;
    cp64 = k.cp64;
  } else {
    const ConvTCParams& k = pl.kp;
    kc = k.kc;
    act_box = k.halo ? k.box_w : k.tile_w * k.sw;
    es_w = k.halo ? 1 : k.sw;
    wgt_rows = k.sub_n;
    wgt_rows_last = k.sub_n;
    cp64 = k.cp64;
  }
  if (pl.cm && pl.cp.gather) {
    // gather mode: the raw input as runs of 16-byte groups of 8 values, dims
    // (8, W * C / 8, H, D, N) for NDHWC or (8, W / 8, H, D, N * C) for NCDHW; one box =
    // g_row_bytes / 16 groups of one row
    const ConvCMParams& k = pl.cp;
    const bool cl = p->layout == CONV3D_NDHWC;
    const cuuint64_t row = cl ? (cuuint64_t)p->W * p->Cin : (cuuint64_t)p->W;
    const cuuint64_t gdim[5] = {8, row / 8, (cuuint64_t)p->H, (cuuint64_t)p->D,
                                (cuuint64_t)p->N * (cl ? 1 : p->Cin)};
    const cuuint64_t gstr[4] = {16, row * 2, row * 2 * p->H, row * 2 * p->H * p->D};
    const cuuint32_t box[5] = {8, (cuuint32_t)(k.g_row_bytes / 16), 1, 1, 1};
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    CUresult rg = enc(tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(xin), gdim,
                      gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rg != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
    // the weights are read directly; valid maps of them fill the unused slots
    const cuuint64_t Kt = (cuuint64_t)p->KT * p->KR * p->KS * k.cp64;
    const cuuint64_t gdB[2] = {Kt, (cuuint64_t)p->Cout};
    const cuuint64_t gsB[1] = {Kt * 2};
    const cuuint32_t bxB[2] = {32, (cuuint32_t)k.wgt_rows};
    const cuuint32_t esB[2] = {1, 1};
    rg = enc(tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->w_packed), gdB, gsB,
             bxB, esB, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rg != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
    *tmBLast = *tmB;
    if (half) half->act = half->wgt = half->wgt_last = *tmB;
    return CONV3D_OK;
  }
  // activations: NDHWC bf16, dims (C, W, H, D, N); one box = kc channels x a run of
  // input pixels along W (element stride = the W stride of the convolution)
  const cuuint64_t C = static_cast<cuuint64_t>(pl.Cst);
  cuuint64_t gdimA[5] = {C, (cuuint64_t)p->W, (cuuint64_t)p->H, (cuuint64_t)p->D,
                         (cuuint64_t)p->N};
  cuuint64_t gstrA[4] = {C * 2, C * 2 * p->W, C * 2 * p->W * p->H, C * 2 * p->W * p->H * p->D};
  cuuint32_t boxA[5] = {(cuuint32_t)kc, (cuuint32_t)act_box, 1, 1, 1};
  cuuint32_t esA[5] = {1, (cuuint32_t)es_w, 1, 1, 1};
  if (pl.cm && pl.cp.rows_box) {
    // direct tiles: all rh rows of the tile in one box, rows sh apart
    boxA[2] = (cuuint32_t)(pl.cp.rh * pl.cp.sh);
    esA[2] = (cuuint32_t)pl.cp.sh;
  }
  cuuint32_t rankA = 5;
  if (flat && pl.cm && pl.cp.compact) {
    // the compact form's im2col map keeps the five dimensions (encoded below)
  } else if (flat && pl.cm && pl.cp.flat3) {
    // D, H and W merged into one dimension of D*H*W positions (dims C, D*H*W, 1, N)
    gdimA[1] = (cuuint64_t)p->D * p->H * p->W;
    gdimA[2] = 1;
    gdimA[3] = (cuuint64_t)p->N;
    gstrA[1] = gstrA[3];
    gstrA[2] = gstrA[3];
    rankA = 4;
  } else if (flat) {
    // H and W merged into one dimension of H*W positions (dims C, H*W, D, N)
    gdimA[1] = (cuuint64_t)p->H * p->W;
    gdimA[2] = (cuuint64_t)p->D;
    gdimA[3] = (cuuint64_t)p->N;
    gstrA[1] = gstrA[2];
    gstrA[2] = gstrA[3];
    rankA = 4;
  }
  CUresult r;
  if (flat && pl.cm && pl.cp.compact) {
    // compact volume: an im2col map over (C, W, H, D, N) whose traversal walks W x Ho x
    // Do from (0, 0, -pt); corner arrays in W, H, D order.  Box = kc channels x box_w
    // pixels of the traversal.
    EncodeIm2colFn enc2 = encode_im2col_fn();
    if (!enc2) return CONV3D_ERR_CUDA;
    const int lo[3] = {0, 0, -p->pad[0].before};
    const int up[3] = {0, -(p->KR - 1), p->pad[0].after - (p->KT - 1)};
    const cuuint32_t es1[5] = {1, 1, 1, 1, 1};
    r = enc2(tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(xin), gdimA, gstrA, lo,
             up, (cuuint32_t)kc, (cuuint32_t)act_box, es1, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle_of(kc), CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    r = enc(tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rankA, const_cast<void*>(xin), gdimA, gstrA,
            boxA, esA, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(kc),
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
  // packed weights [Cout][taps * cp64]: one box = kc channels x wgt_rows output channels
  const cuuint64_t Ktot = (cuuint64_t)p->KT * p->KR * p->KS * cp64;
  cuuint64_t gdimB[2] = {Ktot, (cuuint64_t)p->Cout};
  cuuint64_t gstrB[1] = {Ktot * 2};
  cuuint32_t boxB[2] = {(cuuint32_t)kc, (cuuint32_t)wgt_rows};
  cuuint32_t esB[2] = {1, 1};
  r = enc(tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->w_packed), gdimB, gstrB,
          boxB, esB, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(kc),
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
  if (half) {
    // paired last chunks: the same tensors in 32-channel boxes with 64-byte rows
    if (pl.cm && pl.cp.pair) {
      cuuint32_t boxAh[5] = {32, boxA[1], boxA[2], boxA[3], boxA[4]};
      r = enc(&half->act, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rankA, const_cast<void*>(xin), gdimA,
              gstrA, boxAh, esA, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
      const cuuint32_t rows[2] = {(cuuint32_t)wgt_rows, (cuuint32_t)wgt_rows_last};
      CUtensorMap* dst[2] = {&half->wgt, &half->wgt_last};
      for (int i = 0; i < 2; ++i) {
        cuuint32_t boxBh[2] = {32, rows[i]};
        r = enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->w_packed), gdimB,
                gstrB, boxBh, esB, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
      }
    } else {
      half->act = half->wgt = half->wgt_last = *tmB;  // not used
    }
  }
  // the last 128-channel tile: a box of its real rows only
  if (wgt_rows_last == wgt_rows) {
    *tmBLast = *tmB;
    return CONV3D_OK;
  }
  cuuint32_t boxL[2] = {(cuuint32_t)kc, (cuuint32_t)wgt_rows_last};
  r = enc(tmBLast, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p->w_packed), gdimB,
          gstrB, boxL, esB, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_of(kc),
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
  return CONV3D_OK;
}

// Output maps of the bulk-store epilogue, bf16, box 32 channels x 32 pixels along
// W: NDHWC dims (C, W, H, D, N), or NCDHW dims (W, H, D, C, N).
int encode_out_maps(const conv3d_params* p, const Plan& pl, vvc::CmOutMaps* om) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return CONV3D_ERR_CUDA;
  const cuuint64_t C = (cuuint64_t)p->Cout;
  const cuuint64_t Wo = (cuuint64_t)pl.Wo, Ho = (cuuint64_t)pl.Ho, Do = (cuuint64_t)pl.Do;
  const bool cl = p->out_layout == CONV3D_NDHWC;
  const cuuint64_t gdim[5] = {cl ? C : Wo, cl ? Wo : Ho, cl ? Ho : Do, cl ? Do : C,
                              (cuuint64_t)p->N};
  const cuuint64_t gstr[4] = {cl ? C * 2 : Wo * 2, cl ? C * 2 * Wo : Wo * Ho * 2,
                              cl ? C * 2 * Wo * Ho : Wo * Ho * Do * 2, C * 2 * Wo * Ho * Do};
  const cuuint32_t box[5] = {32, cl ? 32u : 1u, 1, cl ? 1u : 32u, 1};
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  auto one_g = [&](void* base, const cuuint64_t* dim, const cuuint64_t* str, CUtensorMap* m) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dim, str, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  auto one = [&](void* base, CUtensorMap* m) { return one_g(base, gdim, gstr, m); };
  if (has_halo(p)) {
    // y holds the output at an offset: om.y views the output inside it (same
    // extents, y's strides), om.yfull the whole haloed tensor
    long long Dy, Hy, Wy;
    y_extent(p, pl.Do, pl.Ho, pl.Wo, &Dy, &Hy, &Wy);
    const cuuint64_t fdim[5] = {C, (cuuint64_t)Wy, (cuuint64_t)Hy, (cuuint64_t)Dy,
                                (cuuint64_t)p->N};
    const cuuint64_t fstr[4] = {C * 2, C * 2 * Wy, C * 2 * Wy * Hy, C * 2 * Wy * Hy * Dy};
    const size_t origin = (((size_t)p->out_halo[0].before * Hy + p->out_halo[1].before) * Wy +
                           p->out_halo[2].before) * C * 2;
    void* inner = static_cast<uint8_t*>(p->y) + origin;
    if (!one_g(inner, gdim, fstr, &om->y) || !one_g(p->y, fdim, fstr, &om->yfull))
      return CONV3D_ERR_CUDA;
  } else {
    if (!one(p->y, &om->y)) return CONV3D_ERR_CUDA;
    om->yfull = om->y;
  }
  om->val = om->y;
  om->conv = om->y;
  for (int k = 0; k < 4; ++k) om->ycls[k] = om->y;
  if (p->input_upsample == 2) {
    // the outputs of parity class k = 2 ph + pw: [N, Do, Ho / 2, Wo / 2, C] at rows
    // 2 h + ph, columns 2 w + pw of y
    const cuuint64_t Hl = Ho / 2, Wl = Wo / 2;
    const cuuint64_t cdim[5] = {C, Wl, Hl, Do, (cuuint64_t)p->N};
    const cuuint64_t cstr[4] = {C * 4, C * 4 * Wo, C * 2 * Wo * Ho, C * 2 * Wo * Ho * Do};
    for (int k = 0; k < 4; ++k) {
      void* base = static_cast<uint8_t*>(p->y) + ((size_t)(k >> 1) * Wo + (k & 1)) * C * 2;
      if (!one_g(base, cdim, cstr, &om->ycls[k])) return CONV3D_ERR_CUDA;
    }
  }
  if ((p->epi & CONV3D_EPI_SAVE_VALUE) && !one(p->value_out, &om->val)) return CONV3D_ERR_CUDA;
  if ((p->epi & CONV3D_EPI_DEBUG_STORE_CONV) && !one(p->conv_out, &om->conv))
    return CONV3D_ERR_CUDA;
  return CONV3D_OK;
}

}  // namespace

extern "C" {

size_t conv3d_packed_weight_bytes(int32_t Cout, int32_t Cin, int32_t KT, int32_t KR,
                                  int32_t KS) {
  if (Cout < 1 || Cin < 1 || KT < 1 || KR < 1 || KS < 1) return 0;
  return (size_t)Cout * KT * KR * KS * (size_t)round_up(Cin, 64) * 2;
}

size_t conv3d_packed_weight_bytes_e4m3(int32_t Cout, int32_t Cin, int32_t KT, int32_t KR,
                                       int32_t KS) {
  if (Cout < 1 || Cin < 1 || KT < 1 || KR < 1 || KS < 1) return 0;
  return (size_t)Cout * KT * KR * KS * (size_t)round_up(Cin, 128);
}

int conv3d_pack_weight_e4m3(const void* w_oitrs, int32_t Cout, int32_t Cin, int32_t KT,
                            int32_t KR, int32_t KS, void* w_packed, conv3d_stream_t stream) {
  if (!w_oitrs || !w_packed) return CONV3D_ERR_INVALID_ARG;
  if (Cout < 1 || Cin < 1 || KT < 1 || KR < 1 || KS < 1) return CONV3D_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w_oitrs) & 15u) || (reinterpret_cast<uintptr_t>(w_packed) & 15u))
    return CONV3D_ERR_MISALIGNED;
  const size_t in_bytes = (size_t)Cout * Cin * KT * KR * KS;
  const size_t out_bytes = conv3d_packed_weight_bytes_e4m3(Cout, Cin, KT, KR, KS);
  Span a{reinterpret_cast<uintptr_t>(w_oitrs), reinterpret_cast<uintptr_t>(w_oitrs) + in_bytes};
  Span b{reinterpret_cast<uintptr_t>(w_packed), reinterpret_cast<uintptr_t>(w_packed) + out_bytes};
  if (overlaps(a, b)) return CONV3D_ERR_OVERLAP;
  cudaError_t err = vvc::launch_pack_weight_u8(w_oitrs, w_packed, Cout, Cin, KT * KR * KS,
                                               reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

int conv3d_pack_weight(const void* w_oitrs, int32_t Cout, int32_t Cin, int32_t KT, int32_t KR,
                       int32_t KS, void* w_packed, conv3d_stream_t stream) {
  if (!w_oitrs || !w_packed) return CONV3D_ERR_INVALID_ARG;
  if (Cout < 1 || Cin < 1 || KT < 1 || KR < 1 || KS < 1) return CONV3D_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w_oitrs) & 15u) || (reinterpret_cast<uintptr_t>(w_packed) & 15u))
    return CONV3D_ERR_MISALIGNED;
  const size_t in_bytes = (size_t)Cout * Cin * KT * KR * KS * 2;
  const size_t out_bytes = conv3d_packed_weight_bytes(Cout, Cin, KT, KR, KS);
  Span a{reinterpret_cast<uintptr_t>(w_oitrs), reinterpret_cast<uintptr_t>(w_oitrs) + in_bytes};
  Span b{reinterpret_cast<uintptr_t>(w_packed), reinterpret_cast<uintptr_t>(w_packed) + out_bytes};
  if (overlaps(a, b)) return CONV3D_ERR_OVERLAP;
  cudaError_t err = vvc::launch_pack_weight(w_oitrs, w_packed, Cout, Cin, KT * KR * KS,
                                            reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

int conv3d_workspace_bytes_ex(const conv3d_params* p, const conv3d_tuning* tuning,
                              size_t* bytes) {
  if (!bytes) return CONV3D_ERR_INVALID_ARG;
  Plan pl;
  const int rc = make_plan(p, tuning, &pl);
  if (rc) return rc;
  *bytes = pl.ws_bytes;
  return CONV3D_OK;
}

int conv3d_workspace_bytes(const conv3d_params* p, size_t* bytes) {
  return conv3d_workspace_bytes_ex(p, nullptr, bytes);
}

int conv3d_launch_count(const conv3d_params* p, const conv3d_tuning* tuning) {
  Plan pl;
  const int rc = make_plan(p, tuning, &pl);
  if (rc) return rc;
  return pl.launches;
}

int conv3d_plan(const conv3d_params* p, const conv3d_tuning* tuning, conv3d_plan_info* info) {
  if (!info) return CONV3D_ERR_INVALID_ARG;
  Plan pl;
  const int rc = make_plan(p, tuning, &pl);
  if (rc) return rc;
  conv3d_plan_info r{};
  if (pl.cm) {
    const ConvCMParams& k = pl.cp;
    r.kernel = 2;
    r.mma_n = k.N;
    r.stages_per_tile = k.stages_total;
    r.k_splits = k.k_splits;
    r.paired = k.pair;
    r.bulk_store = k.tma_store;
    r.flat = k.flat ? (k.flat3 ? (k.compact ? 3 : 2) : 1) : 0;
  } else {
    const ConvTCParams& k = pl.kp;
    r.kernel = 1;
    r.mma_n = k.BN;
    r.stages_per_tile = k.stages_total;
    r.k_splits = k.k_splits;
  }
  r.im2col = pl.im2col ? 1 : ((pl.cm && pl.cp.gather) ? 2 : 0);
  r.launches = pl.launches;
  r.grid = static_cast<int32_t>(pl.grid.x);
  *info = r;
  return CONV3D_OK;
}

// Padded output + cache: the activations at `act` (contiguous [N, Do, Ho, Wo, Cout])
// go to the interiors of planes 2.. of y, the newest frames to the cache tail, and
// the borders and missing history planes are zeroed; nothing else is written.
int place_pad_cache(const conv3d_params* p, const Plan& pl, const void* act, cudaStream_t s) {
  if (!pl.pad_cache) return CONV3D_OK;
  vvc::PadCacheArgs a{};
  a.act = static_cast<const uint16_t*>(act);
  a.a_sh = (long long)pl.Wo * p->Cout;
  a.a_st = a.a_sh * pl.Ho;
  a.a_sn = a.a_st * pl.Do;
  a.prev = nullptr;
  a.padded = static_cast<uint16_t*>(p->y);
  a.cache = static_cast<uint16_t*>(p->cache_out);
  a.N = p->N;
  a.Tc = pl.Do;
  a.Hc = pl.Ho;
  a.Wc = pl.Wo;
  a.C = p->Cout;
  a.P = p->history_frames;
  a.K = std::min(2, pl.Do + p->history_frames);
  a.copy_interior = 1;
  return vvc::launch_pad_cache(a, s) == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

int conv3d_fwd_ex(const conv3d_params* p, const conv3d_tuning* tuning, conv3d_stream_t stream) {
  Plan pl;
  int rc = make_plan(p, tuning, &pl);
  if (rc) return rc;
  rc = check_pointers(p, pl);
  if (rc) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void* xin = p->x;
  uint8_t* ws = static_cast<uint8_t*>(p->workspace);
  // where the kernels write y: the caller's y, or (padded output + cache) the
  // contiguous scratch activations that the last launch places
  void* yk = pl.pad_cache ? static_cast<void*>(ws + pl.pc_off) : p->y;
  conv3d_params pk = *p;
  pk.y = yk;
  const conv3d_params* pm = &pk;  // the convolution the tensor maps describe
  conv3d_params q;
  if (pl.im2col) {
    void* dst = ws + pl.stage_off;
    void* wr = ws + pl.wr_off;
    const int rh = (p->pad[1].mode == CONV3D_PAD_REFLECT && (p->pad[1].before || p->pad[1].after));
    const int rw = (p->pad[2].mode == CONV3D_PAD_REFLECT && (p->pad[2].before || p->pad[2].after));
    if (vvc::launch_im2col_hw(p->x, p->layout, p->N, p->Cin, p->D, p->H, p->W, pl.Ho, pl.Wo,
                              p->KT, p->KR, p->KS, p->stride[1], p->stride[2], p->pad[1].before,
                              p->pad[2].before, rh, rw, pl.Ck, dst, p->w_packed, p->Cout, wr,
                              s) != cudaSuccess)
      return CONV3D_ERR_CUDA;
    q = pl.q;
    q.x = dst;
    q.w_packed = wr;
    q.y = yk;
    pm = &q;
    xin = dst;
  } else if (pl.f8) {
    q = pl.q;
    q.x = p->x;
    q.w_packed = p->w_packed;
    q.y = yk;
    pm = &q;
  } else if (pl.stage) {
    void* dst = ws + pl.stage_off;
    if (vvc::launch_stage_input(p->x, p->layout, p->N, p->Cin, pl.Cst,
                                (long long)p->D * p->H * p->W, dst, s) != cudaSuccess)
      return CONV3D_ERR_CUDA;
    xin = dst;
  }
  CUtensorMap tmA, tmB, tmBLast;
  vvc::CmHalfMaps half;
  rc = encode_maps(pm, pl, xin, &tmA, &tmB, &tmBLast, &half);
  if (rc) return rc;
  float* partial = reinterpret_cast<float*>(ws + pl.partial_off);
  if (pl.cm) {
    ConvCMParams kp = pl.cp;
    kp.epi.y = yk;
    kp.g_wp = static_cast<const uint16_t*>(p->w_packed);
    if (kp.k_splits > 1) kp.partial = partial;
    if (kp.norm) kp.vscratch = reinterpret_cast<uint16_t*>(ws + pl.vscratch_off);
    vvc::CmOutMaps om;
    if (kp.tma_store) {
      rc = encode_out_maps(pm, pl, &om);
      if (rc) return rc;
    } else {
      om.y = om.val = om.conv = om.yfull = tmA;  // not used
    }
    if (vvc::launch_conv_cm(tmA, tmB, tmBLast, om, half, kp, static_cast<int>(pl.grid.x), pl.smem,
                            s) !=
        cudaSuccess)
      return CONV3D_ERR_CUDA;
    if (kp.k_splits > 1 &&
        vvc::launch_splitk_epilogue(partial, kp.k_splits, kp.M_total, kp.epi, s) != cudaSuccess)
      return CONV3D_ERR_CUDA;
    return place_pad_cache(p, pl, yk, s);
  }
  ConvTCParams kp = pl.kp;
  kp.epi.y = yk;
  if (kp.k_splits > 1) kp.partial = partial;
  if (vvc::launch_conv_tc(tmA, tmB, kp, pl.grid, pl.smem, s) != cudaSuccess)
    return CONV3D_ERR_CUDA;
  if (kp.k_splits > 1 &&
      vvc::launch_splitk_epilogue(partial, kp.k_splits, kp.M_total, kp.epi, s) != cudaSuccess)
    return CONV3D_ERR_CUDA;
  return place_pad_cache(p, pl, yk, s);
}

int conv3d_fwd(const conv3d_params* p, conv3d_stream_t stream) {
  return conv3d_fwd_ex(p, nullptr, stream);
}

int l2norm_silu(const void* x, int64_t rows, int32_t C, const float* input_bias,
                const void* residual, const float* residual_bias, const float* gamma, void* y,
                void* value_out, conv3d_stream_t stream) {
  if (!x || !y || !gamma || rows < 1 || C < 1) return CONV3D_ERR_INVALID_ARG;
  if (rows > 0x7fffffffLL) return CONV3D_ERR_UNSUPPORTED;
  if (residual_bias && !residual) return CONV3D_ERR_INVALID_ARG;
  auto mis = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u); };
  if (mis(x) || mis(y) || mis(input_bias) || mis(residual) || mis(residual_bias) || mis(gamma) ||
      mis(value_out))
    return CONV3D_ERR_MISALIGNED;
  const size_t tb = (size_t)rows * C * 2;
  auto span = [](const void* q, size_t bytes) {
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(q);
    s.hi = q ? s.lo + bytes : s.lo;
    return s;
  };
  const Span in[] = {span(x, tb), span(input_bias, (size_t)C * 4), span(residual, tb),
                     span(residual_bias, (size_t)C * 4), span(gamma, (size_t)C * 4)};
  const Span out[] = {span(y, tb), span(value_out, tb)};
  for (const Span& o : out)
    for (const Span& i : in)
      if (overlaps(o, i)) return CONV3D_ERR_OVERLAP;
  if (overlaps(out[0], out[1])) return CONV3D_ERR_OVERLAP;
  EpiParams e{};
  e.y = y;
  e.out_layout = vvc::LAYOUT_NDHWC;
  e.N = 1;
  e.Cout = C;
  e.Do = 1;
  e.Ho = 1;
  e.Wo = static_cast<int>(rows);
  e.flags = vvc::EPI_L2NORM_SILU | (input_bias ? vvc::EPI_BIAS : 0u) |
            (residual ? vvc::EPI_RESIDUAL : 0u) | (residual_bias ? vvc::EPI_RESIDUAL_BIAS : 0u) |
            (value_out ? vvc::EPI_SAVE_VALUE : 0u);
  e.bias = input_bias;
  e.residual = static_cast<const uint16_t*>(residual);
  e.rbias = residual_bias;
  e.gamma = gamma;
  e.value_out = static_cast<uint16_t*>(value_out);
  e.sqrt_c = std::sqrt(static_cast<float>(C));
  cudaError_t err = vvc::launch_l2norm_silu(x, rows, e, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

int l2norm_silu_pad(const void* x, int32_t N, int32_t T, int32_t H, int32_t W, int32_t C,
                    const float* input_bias, const void* residual, const float* residual_bias,
                    const float* gamma, const void* previous, int32_t history_frames,
                    void* padded_out, void* cache_out, void* value_out,
                    conv3d_stream_t stream) {
  if (!x || !gamma || !padded_out || !cache_out || N < 1 || T < 1 || H < 1 || W < 1 || C < 8 ||
      C % 8 != 0 || history_frames < 0 || history_frames > 2 ||
      (history_frames > 0) != (previous != nullptr) || (residual_bias && !residual))
    return CONV3D_ERR_INVALID_ARG;
  const long long rows = (long long)N * T * H * W;
  const long long padded_rows = (long long)N * (T + 2) * (H + 2) * (W + 2);
  if (padded_rows > 0x7fffffffLL) return CONV3D_ERR_UNSUPPORTED;
  auto mis = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u); };
  if (mis(x) || mis(input_bias) || mis(residual) || mis(residual_bias) || mis(gamma) ||
      mis(previous) || mis(padded_out) || mis(cache_out) || mis(value_out))
    return CONV3D_ERR_MISALIGNED;
  const int K = std::min(2, T + history_frames);
  const size_t tb = (size_t)rows * C * 2;
  auto span = [](const void* q, size_t bytes) {
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(q);
    s.hi = q ? s.lo + bytes : s.lo;
    return s;
  };
  const Span in[] = {span(x, tb), span(input_bias, (size_t)C * 4), span(residual, tb),
                     span(residual_bias, (size_t)C * 4), span(gamma, (size_t)C * 4),
                     span(previous, (size_t)N * history_frames * H * W * C * 2)};
  const Span out[] = {span(padded_out, (size_t)padded_rows * C * 2),
                      span(cache_out, (size_t)N * K * H * W * C * 2), span(value_out, tb)};
  for (size_t i = 0; i < sizeof(out) / sizeof(out[0]); ++i) {
    for (const Span& sp : in)
      if (overlaps(out[i], sp)) return CONV3D_ERR_OVERLAP;
    for (size_t j = i + 1; j < sizeof(out) / sizeof(out[0]); ++j)
      if (overlaps(out[i], out[j])) return CONV3D_ERR_OVERLAP;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // 1: the post-operations, each row written to its padded interior position
  EpiParams e{};
  e.y = padded_out;
  e.out_layout = vvc::LAYOUT_NDHWC;
  e.N = 1;
  e.Cout = C;
  e.Do = e.Ho = e.Wo = 1;
  e.flags = vvc::EPI_L2NORM_SILU | (input_bias ? vvc::EPI_BIAS : 0u) |
            (residual ? vvc::EPI_RESIDUAL : 0u) | (residual_bias ? vvc::EPI_RESIDUAL_BIAS : 0u) |
            (value_out ? vvc::EPI_SAVE_VALUE : 0u);
  e.bias = input_bias;
  e.residual = static_cast<const uint16_t*>(residual);
  e.rbias = residual_bias;
  e.gamma = gamma;
  e.value_out = static_cast<uint16_t*>(value_out);
  e.sqrt_c = std::sqrt(static_cast<float>(C));
  if (vvc::launch_l2norm_silu_pad(x, N, T, H, W, e, s) != cudaSuccess) return CONV3D_ERR_CUDA;
  // 2: borders, missing history planes, history copies and the cache, the
  // activations read back from the padded interiors
  vvc::PadCacheArgs a{};
  const long long Wp = W + 2, Hp = H + 2;
  a.act = static_cast<const uint16_t*>(padded_out) + ((2 * Hp + 1) * Wp + 1) * C;
  a.a_sh = Wp * C;
  a.a_st = Hp * Wp * C;
  a.a_sn = (T + 2LL) * Hp * Wp * C;
  a.prev = static_cast<const uint16_t*>(previous);
  a.padded = static_cast<uint16_t*>(padded_out);
  a.cache = static_cast<uint16_t*>(cache_out);
  a.N = N;
  a.Tc = T;
  a.Hc = H;
  a.Wc = W;
  a.C = C;
  a.P = history_frames;
  a.K = K;
  a.copy_interior = 0;
  return vvc::launch_pad_cache(a, s) == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

int conv3d_causal_pack(const void* x, const int64_t* x_strides, int32_t N, int32_t C, int32_t T,
                       int32_t H, int32_t W, const void* previous, int32_t history_frames,
                       void* padded, int32_t Cp, void* cache_out, conv3d_stream_t stream) {
  if (!x || !x_strides || !padded || !cache_out || N < 1 || C < 1 || T < 1 || H < 1 ||
      W < 1 || Cp < C || Cp % 8 != 0 || Cp > 256 || history_frames < 0 || history_frames > 2 ||
      (history_frames > 0) != (previous != nullptr))
    return CONV3D_ERR_INVALID_ARG;
  const int64_t dims[5] = {N, C, T, H, W};
  long long x_last = 0;  // element offset of the chunk's last element
  for (int i = 0; i < 5; ++i) {
    if (x_strides[i] < 0) return CONV3D_ERR_INVALID_ARG;
    x_last += (long long)(dims[i] - 1) * x_strides[i];
  }
  const long long padded_px = (long long)N * (T + 2) * (H + 2) * (W + 2);
  const int K = std::min(2, T + history_frames);
  const long long cache_px = (long long)N * K * H * W;
  if (padded_px > (1LL << 40) / Cp || x_last > (1LL << 42)) return CONV3D_ERR_UNSUPPORTED;
  const uintptr_t ax = reinterpret_cast<uintptr_t>(x);
  if ((ax & 1u) || (reinterpret_cast<uintptr_t>(previous) & 7u) ||
      (reinterpret_cast<uintptr_t>(padded) & 15u) || (reinterpret_cast<uintptr_t>(cache_out) & 15u))
    return CONV3D_ERR_MISALIGNED;
  auto span = [](const void* q, size_t bytes) {
    Span sp;
    sp.lo = reinterpret_cast<uintptr_t>(q);
    sp.hi = q ? sp.lo + bytes : sp.lo;
    return sp;
  };
  const Span in[] = {span(x, (size_t)(x_last + 1) * 2),
                     span(previous, (size_t)N * history_frames * H * W * C * 2)};
  const Span out[] = {span(padded, (size_t)padded_px * Cp * 2),
                      span(cache_out, (size_t)cache_px * C * 2)};
  for (const Span& o : out)
    for (const Span& sp : in)
      if (overlaps(o, sp)) return CONV3D_ERR_OVERLAP;
  if (overlaps(out[0], out[1])) return CONV3D_ERR_OVERLAP;
  vvc::CausalPackArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.sx_n = x_strides[0];
  a.sx_c = x_strides[1];
  a.sx_t = x_strides[2];
  a.sx_h = x_strides[3];
  a.sx_w = x_strides[4];
  a.prev = static_cast<const uint16_t*>(previous);
  a.padded = static_cast<uint16_t*>(padded);
  a.cache = static_cast<uint16_t*>(cache_out);
  a.N = N;
  a.C = C;
  a.Cp = Cp;
  a.T = T;
  a.H = H;
  a.W = W;
  a.P = history_frames;
  a.K = K;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  return vvc::launch_causal_pack(a, s) == cudaSuccess ? CONV3D_OK : CONV3D_ERR_CUDA;
}

namespace {
// Geometry of a GroupNorm call; false when the shape is not supported.
bool group_norm_shape(int32_t N, int32_t D, int32_t H, int32_t W, int32_t C, int32_t groups,
                      int32_t time_isolated, vvc::GroupNormArgs* a, int* threads) {
  if (N < 1 || D < 1 || H < 1 || W < 1 || C < 8 || C > 2048 || C % 8 != 0 || groups < 1 ||
      C % groups != 0)
    return false;
  const long long slices = time_isolated ? (long long)N * D : (long long)N;
  const long long P = time_isolated ? (long long)H * W : (long long)D * H * W;
  if (slices > 65535 || P * C > (1LL << 40)) return false;
  long long chunk = 0;
  int chunks = 0;
  vvc::group_norm_geometry(C, P, threads, &chunk, &chunks);
  a->P = P;
  a->chunk = chunk;
  a->chunks = chunks;
  a->slices = static_cast<int>(slices);
  a->C = C;
  a->groups = groups;
  return true;
}
}  // namespace

size_t group_norm_workspace_bytes(int32_t N, int32_t D, int32_t H, int32_t W, int32_t C,
                                  int32_t groups, int32_t time_isolated) {
  vvc::GroupNormArgs a{};
  int threads = 0;
  if (!group_norm_shape(N, D, H, W, C, groups, time_isolated, &a, &threads)) return 0;
  return (size_t)a.slices * a.chunks * a.groups * sizeof(double2);
}

int group_norm_silu(const void* x, int32_t N, int32_t D, int32_t H, int32_t W, int32_t C,
                    int32_t groups, int32_t time_isolated, float eps, const float* gamma,
                    const float* beta, int32_t silu, void* y, void* workspace,
                    size_t workspace_bytes, conv3d_stream_t stream) {
  vvc::GroupNormArgs a{};
  int threads = 0;
  if (!x || !y || !workspace || !(eps >= 0.0f) || eps > 1e30f ||
      !group_norm_shape(N, D, H, W, C, groups, time_isolated, &a, &threads))
    return CONV3D_ERR_INVALID_ARG;
  auto mis = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u); };
  if (mis(x) || mis(y) || mis(gamma) || mis(beta) || mis(workspace)) return CONV3D_ERR_MISALIGNED;
  const size_t need = (size_t)a.slices * a.chunks * a.groups * sizeof(double2);
  if (workspace_bytes < need) return CONV3D_ERR_WORKSPACE;
  const size_t tb = (size_t)N * D * H * W * C * 2;
  auto span = [](const void* q, size_t bytes) {
    Span s;
    s.lo = reinterpret_cast<uintptr_t>(q);
    s.hi = q ? s.lo + bytes : s.lo;
    return s;
  };
  const Span in[] = {span(x, tb), span(gamma, (size_t)C * 4), span(beta, (size_t)C * 4)};
  const Span out[] = {span(y, tb), span(workspace, need)};
  for (size_t i = 0; i < 2; ++i) {
    for (const Span& sp : in)
      if (overlaps(out[i], sp)) return CONV3D_ERR_OVERLAP;
  }
  if (overlaps(out[0], out[1])) return CONV3D_ERR_OVERLAP;
  a.x = static_cast<const uint16_t*>(x);
  a.y = static_cast<uint16_t*>(y);
  a.gamma = gamma;
  a.beta = beta;
  a.partial = static_cast<double2*>(workspace);
  a.silu = silu ? 1 : 0;
  a.eps = eps;
  return vvc::launch_group_norm(a, threads, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? CONV3D_OK
             : CONV3D_ERR_CUDA;
}

int conv3d_get_device_status(int32_t* status, conv3d_stream_t stream) {
  if (!status) return CONV3D_ERR_INVALID_ARG;
  int v = 0, w = 0;
  if (vvc::conv_status_read_clear(&v, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CONV3D_ERR_CUDA;
  if (vvc::conv_cm_status_read_clear(&w) != cudaSuccess) return CONV3D_ERR_CUDA;
  *status = v ? v : w;
  return CONV3D_OK;
}

const char* conv3d_status_string(int status) {
  switch (status) {
    case CONV3D_OK: return "ok";
    case CONV3D_ERR_INVALID_ARG: return "invalid argument";
    case CONV3D_ERR_UNSUPPORTED: return "unsupported configuration";
    case CONV3D_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case CONV3D_ERR_OVERLAP: return "output or workspace overlaps another buffer";
    case CONV3D_ERR_WORKSPACE: return "workspace missing or too small";
    case CONV3D_ERR_CUDA: return "CUDA error";
    case CONV3D_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case CONV3D_ERR_SCRATCH_LIMIT:
      return "call needs more scratch than the allocation-free entry point holds (16 MiB)";
    default: return "unknown status";
  }
}

int conv3d_version(void) { return 320; }

}  // extern "C"

extern "C" size_t conv3d_struct_size(int which) {
  switch (which) {
    case 0: return sizeof(conv3d_params);
    case 1: return sizeof(conv3d_tuning);
    case 2: return sizeof(conv3d_pad);
    case 3: return sizeof(conv3d_plan_info);
    default: return 0;
  }
}

// ---- allocation-free variant of conv3d_fwd -----------------------------------------
//
// Some callers cannot allocate device memory at the point where they run a
// convolution: code that only receives pre-allocated tensors from a host
// framework, allocators that forbid allocation inside a timed or latency-critical
// region, or embedders whose memory is fully reserved up front.  For them the
// scratch that conv3d_fwd takes from the caller's workspace (the channels-last
// staging copy of the input, the gathered taps and repacked weights of a narrow
// input, the split-reduction partial sums, the fused norm's value rows and the
// contiguous activations of the padded output + cache) lives instead in one
// file-scope device array that the CUDA module holds from load until exit.
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, resolved once per device and context.  In
// host code the array's name is only a host-side stand-in, so the address must
// come from cudaGetSymbolAddress with that device current.  A device reset
// destroys the context and may reload the module elsewhere, so each cached
// address is kept with the context it was resolved in and looked up again when
// the current context differs.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
  }
  return fn;
}

struct ScratchSlot {
  CUcontext ctx;
  void* ptr;
};
ScratchSlot g_scratch_slot[vvc::kMaxDevices] = {};
std::mutex g_scratch_mu;

int static_scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= vvc::kMaxDevices)
    return CONV3D_ERR_CUDA;
  CtxGetCurrentFn get = ctx_get_current_fn();
  CUcontext ctx = nullptr;
  if (!get || get(&ctx) != CUDA_SUCCESS) return CONV3D_ERR_CUDA;
  if (!ctx) {
    // the runtime has not made this thread's context current yet; the symbol
    // lookup does (it initialises the device's primary context)
    void* tmp = nullptr;
    if (cudaGetSymbolAddress(&tmp, g_static_scratch) != cudaSuccess) return CONV3D_ERR_CUDA;
    if (get(&ctx) != CUDA_SUCCESS || !ctx) return CONV3D_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& slot = g_scratch_slot[dev];
  if (slot.ptr == nullptr || slot.ctx != ctx) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr)
      return CONV3D_ERR_CUDA;
    slot.ctx = ctx;
    slot.ptr = ptr;
  }
  *out = slot.ptr;
  return CONV3D_OK;
}

}  // namespace

extern "C" int conv3d_fwd_static_scratch(const conv3d_params* p, conv3d_stream_t stream) {
  if (!p) return CONV3D_ERR_INVALID_ARG;
  Plan pl;
  int rc = make_plan(p, nullptr, &pl);
  if (rc) return rc;
  conv3d_tuning tu{};
  const conv3d_tuning* tp = nullptr;
  if (pl.ws_bytes > kStaticScratchBytes && pl.cm && pl.cp.norm) {
    // the fused-norm value rows do not fit: pixel-major tiles need none
    tu.kernel = 1;
    tp = &tu;
    rc = make_plan(p, tp, &pl);
    if (rc) return rc;
  }
  if (pl.ws_bytes > kStaticScratchBytes) return CONV3D_ERR_SCRATCH_LIMIT;
  conv3d_params q = *p;
  if (pl.ws_bytes > 0) {
    void* scratch = nullptr;
    rc = static_scratch_for_current_device(&scratch);
    if (rc) return rc;
    q.workspace = scratch;
    q.workspace_bytes = kStaticScratchBytes;
  }
  // Nothing in the scratch needs to start at zero: the staging copy, the gathered
  // taps and repacked weights, every partial sum, the fused-norm value rows and
  // the padded-output activations are written before they are read within the
  // same call.
  return conv3d_fwd_ex(&q, tp, stream);
}
