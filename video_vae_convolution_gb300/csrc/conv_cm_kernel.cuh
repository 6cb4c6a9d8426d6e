// Channel-major implicit-GEMM bf16 convolution on the sm_103a tensor cores.
//
// Same GEMM as conv_tc.cu (ROCm/FlyDSL issue "[Feature]: conv3d_implicit —
// accept and emit NDHWC ...": output pixels x output channels x (taps *
// input channels)), but with the operands swapped so that every MMA is as wide
// as the hardware allows: the accumulator is D[channel][pixel] in TMEM, each
// tcgen05.mma is M = 128 output channels (packed weights, cuDNN frontend doc
// "Fused Conv3D + Bias + Residual + RMSNorm + SiLU", "Weight Packing") by
// N = up to 256 output pixels (activations) by K = 16.  On sm_103a an MMA's
// cost grows with N (M = 128: about 64 cycles at N = 128, 128 at N = 256 when the
// issuing thread keeps up), so the tensor pipe stays busy with N = 256 even when
// the layer has only 96 or 128 output channels; what it cannot hide is the
// issuing thread's own work between MMAs, so the common stage shapes issue from
// straight-line code.
//
// Persistent CTAs walk a static list of tiles (128 channels x one pixel tile,
// times a slice of the reduction when it is split).  A pixel tile is either one
// run of up to 256 output pixels of one output row (halo mode, stride 1 along W:
// one TMA run of tw + KS - 1 input pixels serves all KS taps as shifted views),
// 256 consecutive positions of the flattened H*W plane (flat mode), or rh rows
// of tw pixels (direct mode: one TMA box per row and tap, element stride = conv
// stride).  Channel chunks are 64 wide (128-byte swizzled rows); with the paired
// schedule the last 32-channel chunks of two tap pairs share a stage as 64-byte
// rows.  The accumulator is double buffered in TMEM so the epilogue of one tile
// runs under the MMAs of the next.
//
// Warp roles (128 + 128 G threads): 0 activation producer, 1 MMA issuer + TMEM
// owner, 2 reflect-W patcher, 3 weight producer, 4.. epilogue in G warpgroups
// (G = 2 or 3) that take every G-th 32-pixel column block (a warp reads the TMEM
// lane quarter warp % 4: thread = output channel).  Output blocks on one output
// row go out through bulk tensor stores, the others through per-thread stores.
// Waits are bounded; a time-out records CONV3D_ERR_DEVICE_TIMEOUT.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "epilogue.cuh"
#include "epilogue_cm.cuh"
#include "internal.h"
#include "kernel_common.cuh"
#include "ptx.cuh"

namespace vvc {

// Device status word of the translation unit that instantiates the kernel (each
// unit has its own; the library reads and clears all of them).
static __device__ int g_conv_cm_status = 0;

namespace {

constexpr int kWarpProducer = 0;
constexpr int kWarpMMA = 1;
constexpr int kWarpPatch = 2;
constexpr int kWarpWgt = 3;
constexpr int kWarpEpi0 = 4;
constexpr int kMaxThreads = 512;  // 4 role warps + up to 3 epilogue warpgroups

template <int V>
struct IntC {
  static constexpr int value = V;
};

struct TileCoord {
  int ct, cls, split, twi, thi, od, nb;
};

// Tile index, fastest first: channel tile, split, output depth, W tile, H tile,
// batch (with d_cheap, the output depths past the first d_cheap ones, then those).  CTAs run consecutive tiles at the same time, so with the output depth
// next to the channel tile they share input rows across all output depths while
// those rows are still in L2 (the 3-D layers read their input from HBM about once).
__device__ __forceinline__ TileCoord decode_tile(const ConvCMParams& p, int tile) {
  TileCoord c;
  c.ct = tile % p.tiles_c;
  tile /= p.tiles_c;
  c.cls = 0;
  if (p.ncls > 1) {  // parity class of an x2 upsampled input
    c.cls = tile % p.ncls;
    tile /= p.ncls;
  }
  c.split = tile % p.k_splits;
  tile /= p.k_splits;
  if (p.d_cheap) {
    // the tiles of the first d_cheap output frames (shorter: they leave out temporal taps
    // that read only padding) come after all others, so that every CTA's last round
    // takes some of them
    const int full = p.tiles_d - p.d_cheap;
    const int n_full = full * p.tiles_w * p.tiles_h * p.epi.N;
    if (tile < n_full) {
      c.od = p.d_cheap + tile % full;
      tile /= full;
    } else {
      tile -= n_full;
      c.od = tile % p.d_cheap;
      tile /= p.d_cheap;
    }
  } else {
    c.od = tile % p.tiles_d;
    tile /= p.tiles_d;
  }
  c.twi = tile % p.tiles_w;
  tile /= p.tiles_w;
  c.thi = tile % p.tiles_h;
  c.nb = tile / p.tiles_h;
  return c;
}

struct StageCoord {
  int t, r, sblk, ch;
  int pi, np;  // paired schedule: tap pair index; 0 = full chunk, else pairs in the stage
};

__device__ __forceinline__ StageCoord decode_stage(const ConvCMParams& p, int it) {
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

// e4m3 operands: the accumulator times the call's scale, in place (fp32, round to
// nearest), before anything rounds it to bf16 or writes it as a partial sum.
template <bool kF8>
__device__ __forceinline__ void scale_acc(uint32_t (&r)[32], float s) {
  if constexpr (kF8) {
#pragma unroll
    for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), s));
  }
}

// Stage after c, in the order decode_stage numbers them (no divisions: the
// issuing threads sit on the load-latency path).
__device__ __forceinline__ void next_stage(const ConvCMParams& p, StageCoord& c) {
  if (++c.ch < p.n_chunks) return;
  c.ch = 0;
  if (!p.halo) {
    if (++c.sblk < p.KS) return;
    c.sblk = 0;
  }
  if (++c.r < p.KR) return;
  c.r = 0;
  ++c.t;
}

// Paired schedule (ConvCMParams::pair): per group of two tap pairs, the full
// chunks of the first pair, those of the second, then the last chunks of both in
// one stage.  (t, r) are the coordinates of tap pair pi (pi = t * KR + r).
__device__ __forceinline__ void pair_step(const ConvCMParams& p, int& t, int& r) {
  if (++r == p.KR) {
    r = 0;
    ++t;
  }
}

__device__ __forceinline__ StageCoord pair_begin(const ConvCMParams& p) {
  StageCoord c;
  c.t = c.r = c.sblk = c.pi = 0;
  c.ch = p.n_chunks > 1 ? 0 : p.n_chunks - 1;
  c.np = p.n_chunks > 1 ? 0 : min(2, p.n_pairs);
  return c;
}

__device__ __forceinline__ void pair_next(const ConvCMParams& p, StageCoord& c) {
  if (c.np == 0) {
    if (++c.ch < p.n_chunks - 1) return;
    c.ch = 0;
    if ((c.pi & 1) == 0 && c.pi + 1 < p.n_pairs) {  // the group's second pair
      ++c.pi;
      pair_step(p, c.t, c.r);
      return;
    }
    if (c.pi & 1) {  // back to the group's first pair for its last-chunk stage
      --c.pi;
      if (--c.r < 0) {
        c.r = p.KR - 1;
        --c.t;
      }
    }
    c.np = min(2, p.n_pairs - c.pi);
    c.ch = p.n_chunks - 1;
    return;
  }
  c.pi += 2;  // next group
  pair_step(p, c.t, c.r);
  pair_step(p, c.t, c.r);
  c.np = p.n_chunks > 1 ? 0 : min(2, p.n_pairs - c.pi);
  c.ch = p.n_chunks > 1 ? 0 : p.n_chunks - 1;
}

__device__ __forceinline__ void stage_range(const ConvCMParams& p, int split, int& b, int& e) {
  b = split * p.stages_per_split;
  e = min(p.stages_total, b + p.stages_per_split);
}

// The tile's stage range: its split's slice of the reduction, without the stages whose
// temporal tap reads only T padding for every output frame of the tile (the frames next
// to a zero-padded T edge: the causal pad makes taps 0 and 1 of output frame 0 and tap
// 0 of frame 1 pure zeros).  Stages run in (t, r, s, chunk) order, t slowest, so those
// stages are a prefix and a suffix of the range.  A unit left with no stage keeps its
// first one (it reads zeros and yields the zero partial sum).  Not for the paired
// schedule, which orders stages differently, nor the gather mode (its own producers).
template <bool kPair, bool kGather>
__device__ __forceinline__ void tile_stage_range(const ConvCMParams& p, const TileCoord& tc,
                                                 int& b, int& e) {
  stage_range(p, tc.split, b, e);
  if (kPair || kGather || !p.skip_pad) return;
  int f_lo = tc.od, f_hi = tc.od;  // output frames of the tile
  if (p.flat3) {
    const int plane = (p.compact ? p.epi.Ho : p.H) * p.W;
    f_lo = (tc.twi * p.tw) / plane;
    f_hi = (tc.twi * p.tw + p.tw - 1) / plane;
  }
  const int t_min = max(0, p.pt - f_hi * p.st);
  const int t_max = min(p.KT - 1, p.D - 1 + p.pt - f_lo * p.st);
  if (t_min == 0 && t_max == p.KT - 1) return;
  const int s_t = p.stages_total / p.KT;
  const int lo = max(b, t_min * s_t), hi = min(e, (t_max + 1) * s_t);
  if (lo < hi) {
    b = lo;
    e = hi;
  } else {
    e = b + 1;
  }
}

// The CTA's l-th tile, or -1 past its last.  CTAs take units of tpu consecutive
// tiles round-robin (tpu > 1 keeps the channel tiles of a pixel tile together).
__device__ __forceinline__ int cta_tile(const ConvCMParams& p, int l) {
  const int u = l / p.tpu;
  const long long t = ((long long)blockIdx.x + (long long)u * gridDim.x) * p.tpu + (l - u * p.tpu);
  return t < p.num_tiles ? static_cast<int>(t) : -1;
}

}  // namespace

// kPair: the paired last-chunk schedule (ConvCMParams::pair).  kInner: reflect-W
// halo stages whose inner W taps run before the edge patch.  kPM: pixel-major mode.
// kGather: narrow-input gather mode (ConvCMParams::gather).  kHalo: the output goes
// into a haloed tensor (EpiParams::halo).  kUp2: the input is read x2 upsampled
// (ConvCMParams::up2).
// kF8: e4m3 operands (ConvCMParams::f8): kind::f8f6f4 MMAs and the accumulator scale.
// They are template parameters so that the plain instance keeps the shortest
// producer and MMA-issue loops (the per-stage checks of the first two modes cost
// 4-5 % each on layers that use neither).
template <bool kPair, bool kInner, bool kPM, bool kGather, bool kHalo, bool kUp2,
          bool kF8 = false>
__global__ void __launch_bounds__(kMaxThreads, 1)
    conv_cm_kernel(const __grid_constant__ CUtensorMap tmAct,
                   const __grid_constant__ CUtensorMap tmWgt,
                   const __grid_constant__ CUtensorMap tmWgtLast,
                   const __grid_constant__ CmOutMaps om,
                   const __grid_constant__ CmHalfMaps hm,
                   const __grid_constant__ ConvCMParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  const int S = p.stages;
  const uint32_t bars = sbase + p.bar_off;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto ready_bar = [&](int s) { return bars + 8u * (2 * S + s); };
  auto accf_bar = [&](int b) { return bars + 8u * (3 * S + b); };
  auto acce_bar = [&](int b) { return bars + 8u * (3 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (3 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + p.bar_off + 8 * (3 * S + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int swz = swz_code_for_rowbytes(p.row_bytes);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 2);  // activation and weight producers
      mbar_init(empty_bar(s), 1);
      mbar_init(ready_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      mbar_init(acce_bar(b), 4 * p.epi_groups);  // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmAct);
    tma_prefetch_desc(&tmWgt);
    tma_prefetch_desc(&tmWgtLast);
    if (kPair) {
      tma_prefetch_desc(&hm.act);
      tma_prefetch_desc(&hm.wgt);
      tma_prefetch_desc(&hm.wgt_last);
    }
  }
  if (kGather) {
    // Gather mode: the weights of every (channel tile, temporal tap) stay in shared
    // memory for the whole launch, rows of 32 K values k = (r * KS + s) * C + c in
    // 64-byte swizzled rows: [(ct * KT + kt) * 128 + output channel][k].
    uint8_t* wres = smem + p.g_wres_off;
    const int total = p.tiles_c * p.KT * 128 * 32;
    const int ksc = p.KS * p.C;
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
      const int k = i & 31;
      const int row = i >> 5;
      const int co = (row / (128 * p.KT)) * 128 + (row & 127);
      const int kt = (row >> 7) % p.KT;
      uint16_t v = 0;
      if (co < p.epi.Cout && k < p.g_K) {
        const int r = k / ksc, rem = k - r * ksc;
        const int sx = rem / p.C, c = rem - sx * p.C;
        v = p.g_wp[(((long long)co * p.KT + kt) * p.KR * p.KS + r * p.KS + sx) * p.cp64 + c];
      }
      *reinterpret_cast<uint16_t*>(
          wres + swizzle_off(static_cast<uint32_t>(row * 64 + (k >> 3) * 16), 4) + (k & 7) * 2) = v;
    }
    fence_proxy_async_smem();
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

  if (kGather && warp != kWarpMMA && warp < kWarpEpi0) {
    // Gather mode (one stage per temporal tap kt, tiles of one output row):
    // warp 3 lane 0 copies the KR input rows the stage needs (per input channel
    // for NCDHW input) into the stage's raw region with TMA (runs of 16-byte
    // groups; the first group is rounded down to a 16-byte boundary, rows outside
    // the input read zeros); warps 0 and 2 then expand them into the operand rows
    // [pixel][k = (r * KS + s) * C + c] (zero for k >= K and for pixels past the
    // output row; zero or reflect padding along W) and arrive on the full barrier.
    int slot = 0;
    uint32_t phase = 0;
    bool ok = true;
    if (warp == kWarpWgt) {
      if (lane == 0) {
        long long issued = 0;
        for (int l = 0; ok; ++l) {
          const int tile = cta_tile(p, l);
          if (tile < 0) break;
          const TileCoord tc = decode_tile(p, tile);
          const int w0 = tc.twi * p.tw, ho = tc.thi;
          const int g0 = ((w0 - p.pw) * p.g_cpp) >> 3;  // floor: a negative start reads zeros
          int it_b, it_e;
          stage_range(p, tc.split, it_b, it_e);
          for (int it = it_b; it < it_e; ++it) {
            if (!mbar_wait(empty_bar(slot), phase ^ 1u, abort_flag, lim)) {
              ok = false;
              break;
            }
            const uint32_t raw = sbase + p.stage_bytes * slot + p.g_raw_off;
            mbar_arrive_expect_tx(ready_bar(slot), p.tx_bytes);
            const int d_in = tc.od * p.st + it - p.pt;
            int row = 0;
            for (int c = 0; c < p.g_planes; ++c) {
              for (int r = 0; r < p.KR; ++r, ++row) {
                int h_in = ho * p.sh + r - p.ph;
                if (p.reflect_h) h_in = reflect_coord(h_in, p.H);
                tma_load_5d(raw + static_cast<uint32_t>(row * p.g_row_bytes), &tmAct,
                            ready_bar(slot), 0, g0, h_in, d_in, tc.nb * p.g_planes + c);
              }
            }
            ++issued;
            if (++slot == S) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
        // every issued copy lands before the CTA can exit
        for (int s2 = 0; s2 < S; ++s2) {
          const long long k_last = issued - 1 - ((issued - 1 - s2) % S + S) % S;
          if (k_last >= 0)
            wait_no_abort(ready_bar(s2), static_cast<uint32_t>((k_last / S) & 1), lim);
        }
      }
    } else {
      const int gt = (warp == kWarpProducer ? 0 : 32) + lane;  // expansion thread 0..63
      const int cpp = p.g_cpp;                                  // channels per raw pixel
      const int rstride = p.g_row_bytes >> 1;                   // raw row pitch (elements)
      for (int l = 0; ok; ++l) {
        const int tile = cta_tile(p, l);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int w0 = tc.twi * p.tw;
        const int e0 = (((w0 - p.pw) * cpp) >> 3) << 3;  // first raw element's index in the row
        int it_b, it_e;
        stage_range(p, tc.split, it_b, it_e);
        for (int it = it_b; it < it_e; ++it) {
          if (!mbar_wait(ready_bar(slot), phase, abort_flag, lim)) {
            ok = false;
            break;
          }
          uint8_t* opnd = smem + p.stage_bytes * slot;
          const uint16_t* raw = reinterpret_cast<const uint16_t*>(opnd + p.g_raw_off);
          for (int px = gt; px < p.N; px += 64) {
            const int w = w0 + px;
            const bool live = px < p.tw && w < p.epi.Wo;
            // 16-byte group j of the pixel's 64-byte operand row (swizzled)
            auto store_row = [&](const uint32_t (&pk)[16]) {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                *reinterpret_cast<uint4*>(
                    opnd + swizzle_off(static_cast<uint32_t>(px * 64 + j * 16), 4)) =
                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            };
            if (live && p.KR == 3 && p.KS == 3 && p.C == 3) {
              // the RGB 3x3 case with every index known at compile time (registers only)
              uint32_t pk[16];
#pragma unroll
              for (int q = 0; q < 16; ++q) pk[q] = 0u;
              int wi[3];
              bool inw[3];
#pragma unroll
              for (int sx = 0; sx < 3; ++sx) {
                int w_in = w + sx - p.pw;
                bool in = w_in >= 0 && w_in < p.W;
                if (!in && p.reflect_w) {
                  w_in = reflect_coord(w_in, p.W);
                  in = true;
                }
                wi[sx] = w_in;
                inw[sx] = in;
              }
              const bool planes = p.g_planes > 1;
#pragma unroll
              for (int r = 0; r < 3; ++r) {
#pragma unroll
                for (int sx = 0; sx < 3; ++sx) {
#pragma unroll
                  for (int c = 0; c < 3; ++c) {
                    const int k = (r * 3 + sx) * 3 + c;
                    const int row = (planes ? c * 3 : 0) + r;
                    const int e = (planes ? wi[sx] : wi[sx] * 3 + c) - e0;
                    const uint32_t v = inw[sx] ? uint32_t(raw[row * rstride + e]) : 0u;
                    pk[k >> 1] |= v << (16 * (k & 1));
                  }
                }
              }
              store_row(pk);
            } else {
              uint32_t packed[16];
#pragma unroll
              for (int q = 0; q < 16; ++q) packed[q] = 0u;
              if (live) {
                int k = 0;
                for (int r = 0; r < p.KR; ++r) {
                  for (int sx = 0; sx < p.KS; ++sx) {
                    int w_in = w + sx - p.pw;
                    bool in = w_in >= 0 && w_in < p.W;
                    if (!in && p.reflect_w) {
                      w_in = reflect_coord(w_in, p.W);
                      in = true;
                    }
                    for (int c = 0; c < p.C; ++c, ++k) {
                      uint32_t v = 0u;
                      if (in) {
                        const int row = (p.g_planes > 1 ? c * p.KR : 0) + r;
                        const int e = (p.g_planes > 1 ? w_in : w_in * cpp + c) - e0;
                        v = raw[row * rstride + e];
                      }
                      packed[k >> 1] |= v << (16 * (k & 1));
                    }
                  }
                }
              }
              store_row(packed);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(full_bar(slot));
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp == kWarpProducer || warp == kWarpWgt) {
    // Two producers issue each stage in parallel, each after its own wait on the
    // slot: warp 0 the activation runs, warp 3 the weight boxes.
    const bool act_role = warp == kWarpProducer;
    if (lane == 0) {
      int slot = 0;
      uint32_t phase = 0;
      long long k_global = 0;   // stage counter across tiles
      long long k_skip = -1;    // stage left unissued by the test aid
      bool ok = true;
      for (int l = 0; ok; ++l) {
        const int tile = cta_tile(p, l);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int w0 = tc.twi * p.tw, h0 = tc.thi * p.rh, c0 = tc.ct * 128;
        // the last channel tile loads only its real weight rows, through its own map
        const bool last_ct = tc.ct == p.tiles_c - 1;
        const CUtensorMap* wmap = last_ct ? &tmWgtLast : &tmWgt;
        const uint32_t tx = act_role ? p.act_tx
                                     : (last_ct ? p.tx_bytes_last : p.tx_bytes) - p.act_tx;
        int it_b, it_e;
        tile_stage_range<kPair, kGather>(p, tc, it_b, it_e);
        StageCoord sc = kPair ? pair_begin(p) : decode_stage(p, it_b);
        // compact volume tiles: the traversal start (w, h, d) of each activation box (one
        // box a stage as planned; two kept for generality); a box that would start past
        // the volume's last position starts there instead (its positions are past the end
        // and never stored), so every start lies inside the map's bounding box
        int cq_w[2] = {0, 0}, cq_h[2] = {0, 0}, cq_d[2] = {0, 0};
        if (p.compact && act_role) {
          const int plane = p.epi.Ho * p.W;
          const int q_last = p.epi.Do * plane - 1;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            const int q = min(w0 + b * p.box_w, q_last);
            cq_d[b] = q / plane;
            const int rem = q - cq_d[b] * plane;
            cq_h[b] = rem / p.W;
            cq_w[b] = rem - cq_h[b] * p.W;
          }
        }
        // weight L2 prefetch (plain schedule): pf runs wpref stages ahead of sc
        const bool pref = !kPair && !act_role && p.wpref > 0;
        StageCoord pf = sc;
        int it_pf = it_b;
        auto prefetch_stage = [&](const StageCoord& c) {
          const int x0 = (c.t * p.KR + c.r) * p.KS * p.cp64 + c.ch * p.kc;
          for (int tl = 0; tl < p.taps_per_stage; ++tl)
            tma_prefetch_l2_2d(wmap, x0 + (p.halo ? tl : c.sblk) * p.cp64, c0);
        };
        if (pref) {
          for (; it_pf < it_e && it_pf < it_b + p.wpref; ++it_pf, next_stage(p, pf))
            prefetch_stage(pf);
        }
        for (int it = it_b; it < it_e; ++it, kPair ? pair_next(p, sc) : next_stage(p, sc)) {
          if (pref && it_pf < it_e) {
            prefetch_stage(pf);
            ++it_pf;
            next_stage(p, pf);
          }
          if (!mbar_wait(empty_bar(slot), phase ^ 1u, abort_flag, lim)) {
            ok = false;
            break;
          }
          const bool skip = (p.inject > 0 && k_global == p.inject - 1);
          if (!skip) {
            const uint32_t full = full_bar(slot);
            const int np = kPair ? sc.np : 0;
            mbar_arrive_expect_tx(full, np == 0 ? tx : (tx >> 1) * static_cast<uint32_t>(np));
            const uint32_t act = sbase + p.stage_bytes * slot;
            const uint32_t wgt = act + p.act_bytes;
            const int d_in = tc.od * p.st + sc.t - p.pt;
            if (np > 0) {
              // last chunks of np tap pairs as 32-channel rows of 64 bytes: pair j's
              // run at act + j * act_bytes / 2, its taps' weights after pair j - 1's
              int tj = sc.t, rj = sc.r;
              for (int j = 0; j < np; ++j) {
                if (j) pair_step(p, tj, rj);
                if (!act_role) {
                  const CUtensorMap* hw = last_ct ? &hm.wgt_last : &hm.wgt;
                  for (int tl = 0; tl < p.KS; ++tl) {
                    const int tap = (tj * p.KR + rj) * p.KS + tl;
                    tma_load_2d(wgt + static_cast<uint32_t>((j * p.KS + tl) * p.wtap_rows * 64), hw,
                                full, tap * p.cp64 + sc.ch * p.kc, c0);
                  }
                  continue;
                }
                const int dj = tc.od * p.st + tj - p.pt;
                const uint32_t aj = act + static_cast<uint32_t>(j) * (p.act_bytes >> 1);
                if (p.flat) {
                  const int q_start = p.flat3 ? w0 + ((tj - p.pt) * p.H + rj - p.ph) * p.W
                                              : w0 + (rj - p.ph) * p.W;
                  for (int b = 0; b < p.nbox; ++b)
                    tma_load_4d(aj + static_cast<uint32_t>(b * p.box_w * 64), &hm.act, full,
                                sc.ch * p.kc, q_start + b * p.box_w, p.flat3 ? 0 : dj, tc.nb);
                } else {
                  for (int i = 0; i < p.rh; ++i) {
                    const int ho = h0 + i;
                    int h_in = ho * p.sh + rj - p.ph;
                    if (p.reflect_h && ho < p.epi.Ho) h_in = reflect_coord(h_in, p.H);
                    for (int b = 0; b < p.nbox; ++b)
                      tma_load_5d(aj + static_cast<uint32_t>((i * p.run_pitch + b * p.box_w) * 64),
                                  &hm.act, full, sc.ch * p.kc, w0 - p.pw + b * p.box_w, h_in, dj,
                                  tc.nb);
                  }
                }
              }
            } else if (!act_role) {
              const int x0 = (sc.t * p.KR + sc.r) * p.KS * p.cp64 + sc.ch * p.kc;
              const uint32_t wstep = static_cast<uint32_t>(p.wtap_rows * p.row_bytes);
              if (p.halo && p.taps_per_stage == 3) {
                // the three W taps of a halo stage: consecutive weight boxes
                tma_load_2d(wgt, wmap, full, x0, c0);
                tma_load_2d(wgt + wstep, wmap, full, x0 + p.cp64, c0);
                tma_load_2d(wgt + 2u * wstep, wmap, full, x0 + 2 * p.cp64, c0);
              } else {
                for (int tl = 0; tl < p.taps_per_stage; ++tl) {
                  const int s = p.halo ? tl : sc.sblk;
                  tma_load_2d(wgt + static_cast<uint32_t>(tl) * wstep, wmap, full,
                              x0 + s * p.cp64, c0);
                }
              }
            } else if (p.flat && p.compact) {
              // compact volume: traversal position (w, h, d) of tap (t, r) reads input
              // frame d - pt + t, row h + r; the KS W taps are consecutive positions of
              // the run
#pragma unroll
              for (int b = 0; b < 2; ++b)
                if (b < p.nbox)
                  tma_load_im2col_5d(act + static_cast<uint32_t>(b * p.box_w * p.row_bytes),
                                     &tmAct, full, sc.ch * p.kc, cq_w[b], cq_h[b],
                                     cq_d[b] - p.pt, tc.nb, 0, static_cast<uint16_t>(sc.r),
                                     static_cast<uint16_t>(sc.t));
            } else if (p.flat) {
              // flattened (H*W) positions: output q reads input q + (r - ph) * W + s;
              // flattened (D*H*W) positions: q + ((t - pt) * H + r - ph) * W + s
              const int q_start = p.flat3 ? w0 + ((sc.t - p.pt) * p.H + sc.r - p.ph) * p.W
                                          : w0 + (sc.r - p.ph) * p.W;
              for (int b = 0; b < p.nbox; ++b)
                tma_load_4d(act + static_cast<uint32_t>(b * p.box_w * p.row_bytes), &tmAct,
                            full, sc.ch * p.kc, q_start + b * p.box_w, p.flat3 ? 0 : d_in,
                            tc.nb);
            } else {
              // one run per output row of the tile, run_pitch rows apart: halo runs
              // of tw + KS - 1 pixels (all KS taps), or tw pixels at one tap
              const int w_start = p.halo ? (w0 - p.pw) : (w0 * p.sw + sc.sblk - p.pw);
              if (p.rows_box) {
                // direct tile: every row of the tile in one copy (rows sh apart)
                tma_load_5d(act, &tmAct, full, sc.ch * p.kc, w_start, h0 * p.sh + sc.r - p.ph,
                            d_in, tc.nb);
              } else for (int i = 0; i < p.rh; ++i) {
                const int ho = h0 + i;
                int h_in = ho * p.sh + sc.r - p.ph;
                // x2 upsampled input: class row offsets (-1, 0, 0) or (0, 0, 1)
                if (kUp2) h_in = ho + ((tc.cls >> 1) ? (sc.r == 2 ? 1 : 0) : (sc.r == 0 ? -1 : 0));
                if (p.reflect_h && ho < p.epi.Ho) h_in = reflect_coord(h_in, p.H);
                for (int b = 0; b < p.nbox; ++b)
                  tma_load_5d(act + static_cast<uint32_t>((i * p.run_pitch + b * p.box_w) *
                                                          p.row_bytes),
                              &tmAct, full, sc.ch * p.kc, w_start + b * p.box_w, h_in, d_in,
                              tc.nb);
              }
            }
          } else {
            k_skip = k_global;
          }
          ++k_global;
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
      // Let every issued copy land before the CTA can exit: in each slot, wait
      // for the phase of the last stage issued into it.
      for (int s = 0; s < S; ++s) {
        long long k_last = k_global - 1 - ((k_global - 1 - s) % S + S) % S;
        if (k_last == k_skip) k_last -= S;
        if (k_last >= 0)
          wait_no_abort(full_bar(s), static_cast<uint32_t>((k_last / S) & 1), lim);
      }
    }
  } else if (warp == kWarpMMA) {
    if (lane == 0) {
      // channel-major: A = weights (M = 128 channels), B = pixels (N = p.N);
      // pixel-major: A = pixels (M = 128 per half), B = weights (N = p.pm_n)
      const uint32_t idesc = kF8 ? idesc_e4m3_f32(128, p.N) : idesc_bf16_f32(128, kPM ? p.pm_n : p.N);
      const uint32_t sbo = 8u * static_cast<uint32_t>(p.row_bytes);
      // The high descriptor word (stride, version, swizzle) is fixed; operand
      // views differ only in the start-address field (16-byte units).  The
      // swizzle follows absolute address bits, so row-shifted halo views keep
      // base offset 0.
      const uint32_t desc_hi = static_cast<uint32_t>(sdesc(0u, 16u, sbo, swz, 0u) >> 32);
      const uint32_t desc_lo0 = static_cast<uint32_t>(sdesc(0u, 16u, sbo, swz, 0u));
      const uint32_t w_tap_step = static_cast<uint32_t>(p.wtap_rows * p.row_bytes) >> 4;
      const uint32_t half_step = static_cast<uint32_t>(128 * p.row_bytes) >> 4;
      const uint32_t a_tap_step = p.halo ? (static_cast<uint32_t>(p.row_bytes) >> 4) : 0u;
      // paired last-chunk stages: 64-byte rows (64-byte swizzle, 512-byte row groups)
      const uint32_t desc_hi_h = static_cast<uint32_t>(sdesc(0u, 16u, 512u, 4u, 0u) >> 32);
      const uint32_t w_tap_step_h = static_cast<uint32_t>(p.wtap_rows * 64) >> 4;
      const uint32_t act_half_step = (p.act_bytes >> 1) >> 4;
      // Reflect padding along W (at most 1 on each side): for a stored output pixel
      // only tap 0 can read the reflected pixel left of the row and only tap KS - 1
      // the one right of it (the other taps stay inside the row; what they read from
      // the edge rows lands in halo columns that are never stored).  With halo
      // stages the inner taps go first, so the patch overlaps their MMAs.
      constexpr bool inner_first = kInner;
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int local = 0; ok; ++local) {
        const int tile = cta_tile(p, local);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int buf = (p.nbuf == 2) ? (local & 1) : 0;
        const int use = (p.nbuf == 2) ? (local >> 1) : local;
        if (!mbar_wait(acce_bar(buf), static_cast<uint32_t>(use & 1) ^ 1u, abort_flag, lim)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(buf * p.acc_cols);
        int it_b, it_e;
        tile_stage_range<kPair, kGather>(p, tc, it_b, it_e);
        uint32_t acc = 0u;
        int ch = it_b % p.n_chunks;
        StageCoord psc = pair_begin(p);  // paired schedule only
        for (int it = it_b; it < it_e;
             ++it, ch = (ch + 1 == p.n_chunks) ? 0 : ch + 1, kPair ? pair_next(p, psc) : void()) {
          const uint32_t bar =
              (!kGather && p.reflect_w && !inner_first) ? ready_bar(slot) : full_bar(slot);
          if (!mbar_wait(bar, phase, abort_flag, lim)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // K steps of 16 channels that hold real channels: the rest of a
          // chunk beyond C is zero-filled by TMA and contributes nothing.
          const int chs = kPair ? psc.ch : ch;
          const int kk_n = (min(p.kc, p.C - chs * p.kc) + 15) / 16;
          const uint32_t act = sbase + p.stage_bytes * slot;
          const uint32_t b_lo = desc_lo0 + (act >> 4);
          const uint32_t a_lo = desc_lo0 + ((act + p.act_bytes) >> 4);
          if (kGather) {
            // the stage's 32 K values: resident weights of (channel tile, kt) against
            // the expanded rows, 64-byte swizzle
            const uint32_t w_lo =
                desc_lo0 + ((sbase + p.g_wres_off +
                             static_cast<uint32_t>((tc.ct * p.KT + it) * 128 * 64)) >> 4);
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t adesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (w_lo + 2u * kk);
              const uint64_t bdesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (b_lo + 2u * kk);
              mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
              acc = 1u;
            }
          } else if (kPair && psc.np == 2 && p.KS == 3 && kk_n == 2) {
            // the last 32-channel chunks of two tap pairs, 3 W taps: straight-line issue
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
              for (int tl = 0; tl < 3; ++tl) {
                const uint32_t a_t = a_lo + static_cast<uint32_t>(j * 3 + tl) * w_tap_step_h;
                const uint32_t b_t = b_lo + static_cast<uint32_t>(j) * act_half_step + tl * 4u;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (a_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (b_t + 2u * kk);
                  mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
                  acc = 1u;
                }
              }
            }
          } else if (kPair && psc.np > 0) {
            // the last chunks (<= 32 channels) of psc.np tap pairs
            for (int j = 0; j < psc.np; ++j) {
              for (int tl = 0; tl < p.KS; ++tl) {
                const uint32_t a_t = a_lo + static_cast<uint32_t>(j * p.KS + tl) * w_tap_step_h;
                const uint32_t b_t = b_lo + static_cast<uint32_t>(j) * act_half_step + tl * 4u;
                for (int kk = 0; kk < kk_n; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (a_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi_h) << 32) | (b_t + 2u * kk);
                  mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
                  acc = 1u;
                }
              }
            }
          } else if (!kPM) {
            // a full 64-channel chunk (4 K steps) issues from straight-line code
            const bool full4 = kk_n == 4;
            auto issue_tap = [&](int tl) {
              const uint32_t a_t = a_lo + tl * w_tap_step;
              // x2 upsampled input: W taps read the run shifted by (0, 1, 1) or (1, 1, 2)
              const int tsh = kUp2 ? (tl == 1 ? 1 : (tl == 0 ? (tc.cls & 1) : 1 + (tc.cls & 1))) : tl;
              const uint32_t b_t = b_lo + tsh * a_tap_step;
              if (full4) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | (a_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | (b_t + 2u * kk);
                  mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
                  acc = 1u;
                }
                return;
              }
              if (kk_n == 2) {  // a 32-channel last chunk
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | (a_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | (b_t + 2u * kk);
                  mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
                  acc = 1u;
                }
                return;
              }
              for (int kk = 0; kk < kk_n; ++kk) {
                const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | (a_t + 2u * kk);
                const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | (b_t + 2u * kk);
                mma_ss<kF8>(d, adesc, bdesc, idesc, acc);
                acc = 1u;
              }
            };
            if (inner_first) {
              // taps 1 .. KS - 2 read no patched row for a stored output: they run on
              // the landed copies while the patcher fills the reflected edge rows
              for (int tl = 1; tl < p.KS - 1; ++tl) issue_tap(tl);
              if (!mbar_wait(ready_bar(slot), phase, abort_flag, lim)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_tap(0);
              issue_tap(p.KS - 1);
            } else if (p.taps_per_stage == 3) {
              issue_tap(0);
              issue_tap(1);
              issue_tap(2);
            } else {
              for (int tl = 0; tl < p.taps_per_stage; ++tl) issue_tap(tl);
            }
          } else if (p.pm_halves == 2 && p.taps_per_stage == 3 && (kk_n == 4 || kk_n == 2)) {
            // pixel-major, the common stage shapes (two 128-pixel halves, three W taps
            // of a halo run, a full or a 32-channel chunk): straight-line issue
            const uint32_t acc0 = (it == it_b) ? 0u : 1u;
            auto issue_half = [&](int h, auto kk_c) {
              constexpr int KK = decltype(kk_c)::value;
              const uint32_t dh = d + static_cast<uint32_t>(h * p.pm_cols);
#pragma unroll
              for (int tl = 0; tl < 3; ++tl) {
                const uint32_t x_t = b_lo + h * half_step + tl * a_tap_step;  // pixels
                const uint32_t w_t = a_lo + tl * w_tap_step;                   // weights
#pragma unroll
                for (int kk = 0; kk < KK; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | (x_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | (w_t + 2u * kk);
                  mma_ss<kF8>(dh, adesc, bdesc, idesc, (tl | kk) ? 1u : acc0);
                }
              }
            };
            if (kk_n == 4) {
              issue_half(0, IntC<4>{});
              issue_half(1, IntC<4>{});
            } else {
              issue_half(0, IntC<2>{});
              issue_half(1, IntC<2>{});
            }
          } else {
            // each 128-pixel half of the tile accumulates into its own columns
            for (int h = 0; h < p.pm_halves; ++h) {
              const uint32_t dh = d + static_cast<uint32_t>(h * p.pm_cols);
              uint32_t acc_h = (it == it_b) ? 0u : 1u;
              for (int tl = 0; tl < p.taps_per_stage; ++tl) {
                const uint32_t x_t = b_lo + h * half_step + tl * a_tap_step;  // pixels
                const uint32_t w_t = a_lo + tl * w_tap_step;                   // weights
                for (int kk = 0; kk < kk_n; ++kk) {
                  const uint64_t adesc = (static_cast<uint64_t>(desc_hi) << 32) | (x_t + 2u * kk);
                  const uint64_t bdesc = (static_cast<uint64_t>(desc_hi) << 32) | (w_t + 2u * kk);
                  mma_ss<kF8>(dh, adesc, bdesc, idesc, acc_h);
                  acc_h = 1u;
                }
              }
            }
          }
          mma_commit(empty_bar(slot));
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(accf_bar(buf));
      }
      mma_commit(drain_bar);
      wait_no_abort(drain_bar, 0u, lim);
    }
  } else if (warp == kWarpPatch) {
    if (p.reflect_w) {
      // Reflect padding along W (pad 1): element w = -1 takes x[1] and w = W takes
      // x[W - 2]; TMA filled both with zeros.
      int slot = 0;
      uint32_t phase = 0;
      const int es = p.halo ? 1 : p.sw;
      const int step = 2 / es;
      const int runs = p.rh;
      const int run_len = p.nbox * p.box_w;
      const int run_pitch = p.run_pitch;
      const int chunks = p.row_bytes / 16;
      bool ok = true;
      for (int l = 0; ok; ++l) {
        const int tile = cta_tile(p, l);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int w0 = tc.twi * p.tw;
        int it_b, it_e;
        tile_stage_range<kPair, kGather>(p, tc, it_b, it_e);
        StageCoord sc = kPair ? pair_begin(p) : decode_stage(p, it_b);
        for (int it = it_b; it < it_e; ++it, kPair ? pair_next(p, sc) : next_stage(p, sc)) {
          if (!mbar_wait(full_bar(slot), phase, abort_flag, lim)) {
            ok = false;
            break;
          }
          const int w_start = p.halo ? (w0 - p.pw) : (w0 * p.sw + sc.sblk - p.pw);
          int e_left = -1, e_right = -1;
          if (w_start <= -1 && ((-1 - w_start) % es) == 0) {
            const int e = (-1 - w_start) / es;
            if (e + step < run_len) e_left = e;
          }
          if (p.W - w_start >= 0 && ((p.W - w_start) % es) == 0) {
            const int e = (p.W - w_start) / es;
            if (e < run_len && e - step >= 0) e_right = e;
          }
          uint8_t* act = smem + p.stage_bytes * slot;
          const int work = runs * 2 * chunks;
          for (int wi = lane; wi < work; wi += 32) {
            const int ck = wi % chunks;
            const int side = (wi / chunks) & 1;
            const int k = wi / (2 * chunks);
            const int e = side ? e_right : e_left;
            if (e < 0) continue;
            const int src = side ? e - step : e + step;
            copy_swizzled_row(act, k * run_pitch + src, k * run_pitch + e, p.row_bytes, ck, swz);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(ready_bar(slot));
          if (++slot == S) {
            slot = 0;
            phase ^= 1u;
          }
        }
      }
    }
  } else if (warp >= kWarpEpi0) {
    const int q = warp & 3;              // TMEM lane quarter
    const int grp = (warp - kWarpEpi0) >> 2;  // epilogue warpgroup: every G-th 32-column chunk
    const int G = p.epi_groups;
    const int nepi = 128 * G;  // epilogue threads
    // Everything the epilogue reads per element is copied into registers first.
    CmEpi E;
    E.flags = p.epi.flags;
    E.Cout = p.epi.Cout;
    E.Do = p.epi.Do;
    E.Ho = p.epi.Ho;
    E.Wo = p.epi.Wo;
    E.pad = (E.flags & EPI_OUT_PAD_BR) != 0;
    E.Hy = E.Ho + (E.pad ? 1 : 0);
    E.Wy = E.Wo + (E.pad ? 1 : 0);
    E.ndhwc = (p.epi.out_layout == LAYOUT_NDHWC);
    E.split = p.k_splits > 1;
    E.y = static_cast<uint16_t*>(p.epi.y);
    E.res = p.epi.residual;
    E.val = p.epi.value_out;
    E.conv = p.epi.conv_out;
    E.part = p.partial;
    E.bias = p.epi.bias;
    E.rbias = p.epi.rbias;
    E.gamma = p.epi.gamma;
    E.sqrt_c = p.epi.sqrt_c;
    E.M_total = p.M_total;
    E.halo = kHalo;  // compile-time: calls without a halo carry none of its code
    E.up2 = kUp2;
    E.ep = &p.epi;
    float* st = reinterpret_cast<float*>(smem + p.epi_off) + (warp - kWarpEpi0) * kStageFloats;
    const int nbuf = p.nbuf, acc_cols = p.acc_cols, Ncols = p.N;
    auto tile_view = [&](const TileCoord& tc) {
      CmTile t;
      t.nb = tc.nb;
      t.od = tc.od;
      t.split = tc.split;
      t.w0 = tc.twi * p.tw;
      t.h0 = tc.thi * p.rh;
      t.tw = p.tw;
      t.flat = p.flat;
      t.pitch = p.flat ? p.W : p.run_pitch;
      t.npix = p.flat ? p.tw : p.rh * p.run_pitch;
      t.q0 = p.flat ? t.w0 : 0;
      t.hoff = p.flat ? 0 : t.h0;
      t.woff = p.flat ? 0 : t.w0;
      t.jlim = p.flat ? p.W : p.tw;
      t.vrows = p.flat3 ? (p.compact ? p.epi.Ho : p.H) : 0;
      t.cls = tc.cls;
      return t;
    };
    if (kPM) {
      // Pixel-major: thread = one pixel of the 128-pixel half (TMEM lane), columns =
      // output channels; the per-pixel epilogue reads 16 channels at a time.
      for (int local = 0;; ++local) {
        const int tile = cta_tile(p, local);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int buf = (nbuf == 2) ? (local & 1) : 0;
        const int use = (nbuf == 2) ? (local >> 1) : local;
        if (!mbar_wait(accf_bar(buf), static_cast<uint32_t>(use & 1), abort_flag, lim)) break;
        tc_fence_after();
        const CmTile t = tile_view(tc);
        for (int h = grp; h < p.pm_halves; h += G) {
          const int n = h * 128 + q * 32 + lane;
          Pixel px;
          px.n = tc.nb;
          px.d = tc.od;
          const bool in_tile = cm_pixel(t, n, px.h, px.w);
          px.valid = in_tile && n < t.npix && px.h < E.Ho && px.w < E.Wo;
          const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(buf * acc_cols + h * p.pm_cols);
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
                (((long long)px.n * E.Do + px.d) * E.Ho + px.h) * (long long)E.Wo + px.w;
            for (int c = 0; c < E.Cout; c += 16) {
              float v[16];
              load(c, v);
              if (!px.valid) continue;
              float* dst = p.partial + ((long long)tc.split * p.M_total + pix) * E.Cout + c;
              const int cnt = min(16, E.Cout - c);
#pragma unroll
              for (int k = 0; k < 16; ++k)
                if (k < cnt) dst[k] = v[k];
            }
          } else {
            epilogue_pixel(p.epi, px, 0, E.Cout, load);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
      }
    } else if (!p.norm) {
      const bool dbl_stage = (E.flags & EPI_DEBUG_STORE_CONV) == 0;
      int nbulk = 0;  // bulk blocks this warp has staged
      for (int local = 0;; ++local) {
        const int tile = cta_tile(p, local);
        if (tile < 0) break;
        const TileCoord tc = decode_tile(p, tile);
        const int buf = (nbuf == 2) ? (local & 1) : 0;
        const int use = (nbuf == 2) ? (local >> 1) : local;
        if (!mbar_wait(accf_bar(buf), static_cast<uint32_t>(use & 1), abort_flag, lim)) break;
        tc_fence_after();
        const CmTile t = tile_view(tc);
        const int cw = tc.ct * 128 + q * 32;  // first channel of this warp's TMEM lanes
        const bool warp_live = cw < E.Cout;
        const CmChan ch = cm_chan(E, cw, lane);
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                            static_cast<uint32_t>(buf * acc_cols);
        for (int j0 = 32 * grp; j0 < Ncols; j0 += 32 * G) {
          uint32_t r[32];
          tmem_ld32(tb + static_cast<uint32_t>(j0), r);
          tmem_ld_wait();
          if (!warp_live) continue;
          scale_acc<kF8>(r, p.epi.acc_scale);
          if (p.tma_store) {
            const int qq = t.q0 + j0;
            const int ib = qq / t.pitch;
            const int jb = qq - ib * t.pitch;
            const int wr = t.woff + jb;
            int od, hr;  // output frame and row (a tile of the flattened volume spans frames)
            cm_frame_row(t, t.hoff + ib, od, hr);
            const bool in_row = jb + 31 < t.jlim && jb + 31 < t.pitch && j0 + 31 < t.npix &&
                                hr < E.Ho && od < E.Do && wr + 31 < E.Wo;
            const bool bulk_ncdhw = !E.ndhwc && in_row && (wr & 7) == 0;
            const bool bulk_ndhwc = E.ndhwc && in_row;
            // Bulk blocks alternate between the two 2 KB halves of the staging block, so a
            // block waits only for the store before the previous one to have read its half
            // (the debug conv store takes the second half: one half then).  Any other block
            // writes the whole staging block and waits for every store to have read it.
            uint16_t* yt = reinterpret_cast<uint16_t*>(st);
            if (bulk_ncdhw || bulk_ndhwc) {
              if (dbl_stage) {
                yt += (nbulk & 1) * 1024;
                ++nbulk;
                if (lane == 0) bulk_wait_read_1();
              } else if (lane == 0) {
                bulk_wait_read_all();
              }
            } else if (lane == 0) {
              bulk_wait_read_all();
            }
            __syncwarp();
            if (bulk_ncdhw) {
              // NCDHW: the block goes out as [32 channels][32 pixels] bf16, one 64-byte
              // row per thread (its channel), through bulk tensor stores.  The store's
              // innermost coordinate is the output column, so it must be a multiple of 8.
              const bool bias = (E.flags & EPI_BIAS) != 0;
              uint32_t wv[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float a = round_bf16(__uint_as_float(r[2 * j]));
                float b = round_bf16(__uint_as_float(r[2 * j + 1]));
                if (bias) {
                  a = __fadd_rn(a, ch.bc);
                  b = __fadd_rn(b, ch.bc);
                }
                wv[j] = pack_bf16x2(a, b);
              }
              uint4* row = reinterpret_cast<uint4*>(yt + lane * 32);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                row[k] = make_uint4(wv[4 * k], wv[4 * k + 1], wv[4 * k + 2], wv[4 * k + 3]);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_5d(&om.y, smem_u32(yt), wr, hr, od, cw, tc.nb);
                if (E.flags & EPI_SAVE_VALUE)
                  tma_store_5d(&om.val, smem_u32(yt), wr, hr, od, cw, tc.nb);
                bulk_commit_group();
              }
              continue;
            }
            if (bulk_ndhwc) {
              // The 32 pixels are one piece of an output row: the block goes out as
              // [32 pixels][32 channels] bf16 through bulk tensor stores.
              uint16_t* ct = yt + 32 * 32;
              const bool dbg = (E.flags & EPI_DEBUG_STORE_CONV) != 0;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const uint16_t cb = bf16_bits(__uint_as_float(r[j]));
                uint16_t vb = cb;
                if (E.flags & EPI_BIAS) vb = bf16_bits(__fadd_rn(bf16_val(cb), ch.bc));
                yt[j * 32 + lane] = vb;
                if (dbg) ct[j * 32 + lane] = cb;
              }
              fence_proxy_async_smem();
              __syncwarp();
              // haloed y: om.y views the output inside y; the halo rows that copy
              // this block go out through om.yfull (the whole haloed y, so every
              // coordinate is >= 0), zero halo rows and the halo columns beside or
              // reflecting the block's pixels through plain stores
              const int bh = E.halo ? halo_bits(hr, E.Ho, p.epi.h0, p.epi.Hy - E.Ho - p.epi.h0,
                                                p.epi.h_mode)
                                    : 0;
              if (lane == 0) {
                tma_store_5d(kUp2 ? &om.ycls[tc.cls] : &om.y, smem_u32(yt), cw, wr, hr, od, tc.nb);
                if ((bh & 3) == 1)
                  tma_store_5d(&om.yfull, smem_u32(yt), cw, wr + p.epi.w0, p.epi.h0 - 1,
                               od + p.epi.d0, tc.nb);
                if ((bh & 12) == 4)
                  tma_store_5d(&om.yfull, smem_u32(yt), cw, wr + p.epi.w0, E.Ho + p.epi.h0,
                               od + p.epi.d0, tc.nb);
                if (E.flags & EPI_SAVE_VALUE)
                  tma_store_5d(&om.val, smem_u32(yt), cw, wr, hr, od, tc.nb);
                if (dbg) tma_store_5d(&om.conv, smem_u32(ct), cw, wr, hr, od, tc.nb);
                bulk_commit_group();
              }
              // (only blocks next to a border have halo rows or columns to fill)
              if (E.halo && ((bh & 10) || wr <= 1 || wr + 32 >= E.Wo - 1))
                cm_halo_block(p.epi, yt, lane, tc.nb, od, hr, wr, cw, bh);
              continue;
            }
          }
          cm_block(E, t, st, lane, cw, j0, r, ch);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acce_bar(buf));
      }
      // every bulk store of this warp completes before the CTA can exit
      if (p.tma_store && lane == 0) bulk_wait_all();
      __syncwarp();
    } else {
      // Fused L2 norm: pass 1 per channel tile, pass 2 once per pixel tile.  Every
      // epilogue warp runs the same sequence of named barriers: after a failed wait
      // a warp skips the work but keeps taking part, so no barrier is left short.
      const int tid = threadIdx.x - kWarpEpi0 * 32;
      const int Cs = p.norm_cs;
      float* den = reinterpret_cast<float*>(smem + p.norm_off);  // [N]
      uint16_t* scr = p.vscratch + (long long)blockIdx.x * Ncols * Cs;
      bool ok = true;
      int local = 0;
      for (int l0 = 0;; l0 += p.tpu) {
        const int tile0 = cta_tile(p, l0);
        if (tile0 < 0) break;
        const CmTile t = tile_view(decode_tile(p, tile0));
        for (int ct = 0; ct < p.tiles_c; ++ct, ++local) {
          const int buf = (nbuf == 2) ? (local & 1) : 0;
          const int use = (nbuf == 2) ? (local >> 1) : local;
          if (ok && !mbar_wait(accf_bar(buf), static_cast<uint32_t>(use & 1), abort_flag, lim))
            ok = false;
          if (!ok) continue;
          tc_fence_after();
          const int cw = ct * 128 + q * 32;
          const bool warp_live = cw < E.Cout;
          const CmChan ch = cm_chan(E, cw, lane);
          const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                              static_cast<uint32_t>(buf * acc_cols);
          for (int j0 = 32 * grp; j0 < Ncols; j0 += 32 * G) {
            uint32_t r[32];
            tmem_ld32(tb + static_cast<uint32_t>(j0), r);
            tmem_ld_wait();
            scale_acc<kF8>(r, p.epi.acc_scale);
            if (warp_live) cm_norm_pass1(E, t, st, lane, j0, r, scr, Cs, ch);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(buf));
        }
        named_bar_sync(1, nepi);
        if (ok) {
          for (int n = tid; n < Ncols; n += nepi) {
            int h, w;
            const bool pv = cm_pixel(t, n, h, w) && n < t.npix && h < E.Ho && w < E.Wo;
            den[n] = pv ? cm_norm_den(E, scr + (long long)n * Cs) : 1.0f;
          }
        }
        named_bar_sync(1, nepi);
        if (ok) {
          if (E.ndhwc)
            cm_norm_pass2_ndhwc(E, t, tid, nepi, Ncols, scr, Cs, den);
          else
            cm_norm_pass2_ncdhw(E, t, st, lane, warp - kWarpEpi0, 4 * G, Ncols, scr, Cs, den);
        }
        named_bar_sync(1, nepi);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(&g_conv_cm_status, -7);
}

}  // namespace vvc
