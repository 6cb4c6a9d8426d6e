// Implicit-GEMM bf16 convolution on the sm_103a tensor cores (tcgen05 + TMEM),
// fed by TMA from channels-last (NDHWC) activations.
//
// GEMM view ([FlyDSL#993] ROCm/FlyDSL issue "[Feature]: conv3d_implicit —
// accept and emit NDHWC ...", maintainer comment on the split-K and
// splitk==1 paths): M = output pixels, N = output channels, K = taps x input
// channels:
//   acc[m][co] = sum_{t,r,s,ci} x[n, d*st+t-pt, h*sh+r-ph, w*sw+s-pw, ci] * W[co][t][r][s][ci]
// with W packed OTRSI as in the cuDNN frontend doc "Fused Conv3D + Bias +
// Residual + RMSNorm + SiLU", section "Weight Packing".
//
// One CTA computes R M-tiles (each tile_h output rows x tile_w output pixels of
// one (n, d) plane, 128 TMEM lanes) times BN output channels, over a range of
// K stages.  A stage is one (t, r, s-block, channel chunk): the producer warp
// issues one TMA box per output row (a row of input pixels, kc channels, the
// element stride equal to the conv stride) plus the weight boxes; no im2col is
// materialised.  In halo mode (stride 1 along W) a box holds tile_w + KS - 1
// pixels and the KS taps of that row are shifted views of it.  Zero and causal
// padding come from TMA's out-of-bounds fill; reflect padding remaps rows (H)
// and patches the first / last column in shared memory (W) before the MMA.
//
// Warp roles (256 threads): 0 TMA producer, 1 MMA issuer + TMEM owner,
// 2 reflect-W patcher, 4..7 epilogue (one TMEM lane quarter each).  Every
// wait is bounded: on a time-out the CTA records CONV3D_ERR_DEVICE_TIMEOUT in
// a device status word, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace vvc {

__device__ int g_conv_status = 0;

namespace {

constexpr int kWarpProducer = 0;
constexpr int kWarpMMA = 1;
constexpr int kWarpPatch = 2;
constexpr int kWarpEpi0 = 4;

struct StageCoord {
  int t, r, sblk, ch;
};

__device__ __forceinline__ StageCoord decode_stage(const ConvTCParams& p, int it) {
  StageCoord c;
  c.ch = it % p.n_chunks;
  int rest = it / p.n_chunks;
  if (p.halo) {
    c.sblk = 0;
  } else {
    c.sblk = rest % p.KS;
    rest /= p.KS;
  }
  c.r = rest % p.KR;
  c.t = rest / p.KR;
  return c;
}

}  // namespace

__global__ void __launch_bounds__(256, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ ConvTCParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t a_base = sbase;
  const uint32_t b_base = sbase + p.a_stage_bytes * p.stages;
  const uint32_t bars = sbase + p.bar_off;
  const int S = p.stages;
  const uint32_t accum_bar = bars + 8u * (3 * S);
  const uint32_t drain_bar = accum_bar + 8u;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (3 * S + 2));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- tile coordinates -----------------------------------------------------------
  int bx = blockIdx.x;
  const int tw = bx % p.tiles_w;
  bx /= p.tiles_w;
  const int gh = bx % p.groups_h;
  bx /= p.groups_h;
  const int od = bx % p.epi.Do;
  const int nb = bx / p.epi.Do;
  const int wo0 = tw * p.tile_w;
  const int ho0 = gh * p.R * p.tile_h;
  const int n0 = blockIdx.y * p.BN;
  const int split = blockIdx.z;
  const int it_begin = split * p.stages_per_split;
  const int it_end = min(p.stages_total, it_begin + p.stages_per_split);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bars + 8u * s, 1);            // full: producer arrive + TMA bytes
      mbar_init(bars + 8u * (S + s), 1);      // empty: MMA commit
      mbar_init(bars + 8u * (2 * S + s), 1);  // ready: patcher arrive (reflect W)
    }
    mbar_init(accum_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == kWarpMMA) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const unsigned long long lim = p.timeout_ns;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      int k_skip = -1;  // stage left unissued by the test aid
      for (int it = it_begin; it < it_end; ++it) {
        if (!mbar_wait(bars + 8u * (S + slot), phase ^ 1u, abort_flag, lim)) break;
        const StageCoord sc = decode_stage(p, it);
        const bool skip = (p.inject > 0 && it == p.inject - 1);
        if (!skip) {
          const uint32_t full = bars + 8u * slot;
          mbar_arrive_expect_tx(full, p.tx_bytes);
          const int d_in = od * p.st + sc.t - p.pt;
          const int w_start = wo0 * p.sw + sc.sblk - p.pw;
          const uint32_t a_stage = a_base + p.a_stage_bytes * slot;
          for (int j = 0; j < p.R; ++j) {
            for (int i = 0; i < p.tile_h; ++i) {
              const int ho = ho0 + j * p.tile_h + i;
              int h_in = ho * p.sh + sc.r - p.ph;
              if (p.reflect_h && ho < p.epi.Ho) h_in = reflect_coord(h_in, p.H);
              const uint32_t dst =
                  a_stage + static_cast<uint32_t>((j * p.a_tile_rows + i * p.pitch_rows) *
                                                  p.row_bytes);
              tma_load_5d(dst, &tmA, full, sc.ch * p.kc, w_start, h_in, d_in, nb);
            }
          }
          const uint32_t b_stage = b_base + p.b_stage_bytes * slot;
          for (int tl = 0; tl < p.taps_per_stage; ++tl) {
            const int s = p.halo ? tl : sc.sblk;
            const int tap = (sc.t * p.KR + sc.r) * p.KS + s;
            for (int u = 0; u < p.n_sub; ++u) {
              const uint32_t dst =
                  b_stage + static_cast<uint32_t>((tl * p.BN + u * p.sub_n) * p.row_bytes);
              tma_load_2d(dst, &tmB, full, tap * p.cp64 + sc.ch * p.kc, n0 + u * p.sub_n);
            }
          }
        } else {
          k_skip = it - it_begin;
        }
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      // Let every issued copy land before the CTA can exit: in each slot, wait
      // for the phase of the last stage issued into it.
      const int n_it = it_end - it_begin;
      for (int s = 0; s < S; ++s) {
        int k_last = n_it - 1 - ((n_it - 1 - s) % S + S) % S;
        if (k_last == k_skip) k_last -= S;
        if (k_last >= 0)
          wait_no_abort(bars + 8u * s, static_cast<uint32_t>((k_last / S) & 1), lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.sub_n);
      const uint32_t sbo = 8u * static_cast<uint32_t>(p.row_bytes);
      // Descriptors are built once: the high word (stride, version, swizzle) is
      // fixed, and every operand view is the low word plus an offset in 16-byte
      // units.  The swizzle follows absolute shared-memory address bits, so a
      // view shifted by whole rows (the halo taps) keeps base offset 0.
      const uint32_t desc_hi = static_cast<uint32_t>(sdesc(0u, 16u, sbo, p.swz, 0u) >> 32);
      const uint32_t desc_lo0 = static_cast<uint32_t>(sdesc(0u, 16u, sbo, p.swz, 0u));
      const uint32_t a_tile_step = static_cast<uint32_t>(p.a_tile_rows * p.row_bytes) >> 4;
      const uint32_t a_tap_step = p.halo ? (static_cast<uint32_t>(p.row_bytes) >> 4) : 0u;
      const uint32_t b_tap_step = static_cast<uint32_t>(p.BN * p.row_bytes) >> 4;
      const uint32_t b_sub_step = static_cast<uint32_t>(p.sub_n * p.row_bytes) >> 4;
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = it_begin; it < it_end; ++it) {
        const uint32_t bar = p.reflect_w ? (bars + 8u * (2 * S + slot)) : (bars + 8u * slot);
        if (!mbar_wait(bar, phase, abort_flag, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // K steps of 16 channels that hold real channels: the rest of a chunk
        // beyond C is zero-filled by TMA and contributes nothing.
        const int kk_n = (min(p.kc, p.C - (it % p.n_chunks) * p.kc) + 15) / 16;
        const uint32_t a_lo = desc_lo0 + ((a_base + p.a_stage_bytes * slot) >> 4);
        const uint32_t b_lo = desc_lo0 + ((b_base + p.b_stage_bytes * slot) >> 4);
        uint32_t acc = (it == it_begin) ? 0u : 1u;
        for (int tl = 0; tl < p.taps_per_stage; ++tl) {
          const uint32_t a_tl = a_lo + tl * a_tap_step;
          const uint32_t b_tl = b_lo + tl * b_tap_step;
          for (int kk = 0; kk < kk_n; ++kk) {
            uint32_t d = tmem_base;
            uint32_t a_j = a_tl + 2u * kk;  // 32 bytes per K = 16 step
            for (int j = 0; j < p.R; ++j) {
              const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | a_j;
              uint32_t b_u = b_tl + 2u * kk;
              for (int u = 0; u < p.n_sub; ++u) {
                const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | b_u;
                mma_bf16_ss(d + static_cast<uint32_t>(u * p.sub_n), adesc, bdesc, idesc, acc);
                b_u += b_sub_step;
              }
              a_j += a_tile_step;
              d += static_cast<uint32_t>(p.acc_stride);
            }
            acc = 1u;
          }
        }
        mma_commit(bars + 8u * (S + slot));  // frees the slot once these MMAs finish
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(accum_bar);
      mma_commit(drain_bar);
      wait_no_abort(drain_bar, 0u, lim);
    }
  } else if (warp == kWarpPatch) {
    if (p.reflect_w) {
      // Reflect padding along W (pad 1): the element at w = -1 takes x[1] and the
      // element at w = W takes x[W - 2]; TMA filled both with zeros.
      int slot = 0;
      uint32_t phase = 0;
      const int es = p.halo ? 1 : p.sw;
      const int step = 2 / es;
      const int nbox = p.R * p.tile_h;
      const int chunks = p.row_bytes / 16;
      for (int it = it_begin; it < it_end; ++it) {
        if (!mbar_wait(bars + 8u * slot, phase, abort_flag, lim)) break;
        const StageCoord sc = decode_stage(p, it);
        const int w_start = wo0 * p.sw + sc.sblk - p.pw;
        int e_left = -1, e_right = -1;
        if (w_start <= -1 && ((-1 - w_start) % es) == 0) {
          const int e = (-1 - w_start) / es;
          if (e < p.box_w && e + step < p.box_w) e_left = e;
        }
        if (p.W - w_start >= 0 && ((p.W - w_start) % es) == 0) {
          const int e = (p.W - w_start) / es;
          if (e < p.box_w && e - step >= 0) e_right = e;
        }
        uint8_t* a_stage = smem + p.a_stage_bytes * slot;
        const int work = nbox * 2 * chunks;
        for (int wi = lane; wi < work; wi += 32) {
          const int ck = wi % chunks;
          const int side = (wi / chunks) & 1;
          const int bi = wi / (2 * chunks);
          const int e = side ? e_right : e_left;
          if (e < 0) continue;
          const int src_e = side ? e - step : e + step;
          const int j = bi / p.tile_h, i = bi % p.tile_h;
          const uint32_t box_off =
              static_cast<uint32_t>((j * p.a_tile_rows + i * p.pitch_rows) * p.row_bytes);
          const uint32_t so = swizzle_off(static_cast<uint32_t>(src_e * p.row_bytes + ck * 16), p.swz);
          const uint32_t dof = swizzle_off(static_cast<uint32_t>(e * p.row_bytes + ck * 16), p.swz);
          const uint4 val = *reinterpret_cast<const uint4*>(a_stage + box_off + so);
          *reinterpret_cast<uint4*>(a_stage + box_off + dof) = val;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8u * (2 * S + slot));
        if (++slot == S) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const bool got = mbar_wait(accum_bar, 0u, abort_flag, lim);
    if (got) {
      tc_fence_after();
      const EpiParams& e = p.epi;
      const int ce = min(n0 + p.BN, e.Cout);
      for (int j = 0; j < p.R; ++j) {
        const int i = m / p.tile_w;
        const int jw = m % p.tile_w;
        Pixel px;
        px.n = nb;
        px.d = od;
        px.h = ho0 + j * p.tile_h + i;
        px.w = wo0 + jw;
        px.valid = (i < p.tile_h) && (px.h < e.Ho) && (px.w < e.Wo);
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(j * p.acc_stride);
        auto load = [&](int c_rel, float(&v)[16]) {
          uint32_t r[16];
          tmem_ld16(tb + static_cast<uint32_t>(c_rel), r);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(r[k]);
        };
        if (p.k_splits > 1) {
          // fp32 partial sums, NDHWC-flat [split][M][Cout]
          const long long pix =
              (((long long)px.n * e.Do + px.d) * e.Ho + px.h) * (long long)e.Wo + px.w;
          for (int c = n0; c < ce; c += 16) {
            float v[16];
            load(c - n0, v);
            if (!px.valid) continue;
            float* dst = p.partial + ((long long)split * p.M_total + pix) * e.Cout + c;
            const int cnt = min(16, ce - c);
            if (cnt == 16 && (e.Cout % 4) == 0) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                reinterpret_cast<float4*>(dst)[k] =
                    make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
            } else {
              for (int k = 0; k < cnt; ++k) dst[k] = v[k];
            }
          }
        } else {
          epilogue_pixel(e, px, n0, ce, load);
        }
      }
    }
  }

  // ---- teardown ---------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_conv_status, -7);
}

// ---- host side of this translation unit ---------------------------------------------

cudaError_t launch_conv_tc(const CUtensorMap& tmA, const CUtensorMap& tmB, const ConvTCParams& p,
                           dim3 grid, size_t smem_bytes, cudaStream_t stream) {
  static int opted_in[kMaxDevices] = {};
  cudaError_t err = opt_in_smem(conv_tc_kernel, opted_in);
  if (err != cudaSuccess) return err;
  conv_tc_kernel<<<grid, 256, smem_bytes, stream>>>(tmA, tmB, p);
  return cudaGetLastError();
}

cudaError_t conv_status_read_clear(int* status, cudaStream_t stream) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  int v = 0;
  err = cudaMemcpyFromSymbol(&v, g_conv_status, sizeof(int));
  if (err != cudaSuccess) return err;
  *status = v;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_conv_status, &zero, sizeof(int));
}

}  // namespace vvc
