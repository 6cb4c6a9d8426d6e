// Host/device parameter blocks shared by the launcher (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace vvc {

// Largest device ordinal the per-device host caches hold.
constexpr int kMaxDevices = 64;

// Opts a kernel in to the device's full dynamic shared memory, once per device
// (the attribute belongs to the function on the current device).  `done` is the
// kernel's own per-device flag table; concurrent first calls both set the same
// value, which is harmless.
template <class Kernel>
inline cudaError_t opt_in_smem(Kernel kernel, int (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (__atomic_load_n(&done[dev], __ATOMIC_ACQUIRE)) return cudaSuccess;
  int max_optin = 0;
  err = cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
  if (err != cudaSuccess) return err;
  __atomic_store_n(&done[dev], 1, __ATOMIC_RELEASE);
  return cudaSuccess;
}

enum : unsigned {
  EPI_BIAS = 1u,
  EPI_RESIDUAL = 2u,
  EPI_RESIDUAL_BIAS = 4u,
  EPI_L2NORM_SILU = 8u,
  EPI_SAVE_VALUE = 16u,
  EPI_OUT_PAD_BR = 32u,
  EPI_DEBUG_STORE_CONV = 1u << 30,
};

enum : int { LAYOUT_NCDHW = 0, LAYOUT_NDHWC = 1 };

// Where and how the epilogue writes one output pixel's channel row.
struct EpiParams {
  void* y;                 // bf16 output, out_layout, (Ho+1, Wo+1) with OUT_PAD_BR
  int out_layout;
  int N, Cout, Do, Ho, Wo;
  unsigned flags;
  const float* bias;       // [Cout] (BIAS)
  const uint16_t* residual;  // bf16, out_layout, unpadded (RESIDUAL)
  const float* rbias;      // [Cout] (RESIDUAL_BIAS)
  const float* gamma;      // [Cout] (L2NORM_SILU)
  uint16_t* value_out;     // bf16, out_layout, unpadded (SAVE_VALUE)
  uint16_t* conv_out;      // bf16 NDHWC unpadded (DEBUG_STORE_CONV)
  float sqrt_c;            // sqrtf((float)Cout)
  // Output halo (NDHWC y only; halo = 1): y is [N, Dy, Hy, Wy, Cout] with the output
  // at offset (d0, h0, w0).  Along H and W the halo is at most one pixel on a side
  // (before = h0 / w0, after = Hy - Ho - h0 / Wy - Wo - w0), filled by reflection
  // (mode 2: halo -1 takes row 1, halo Ho takes row Ho - 2) or with zeros (mode 1);
  // the d0 leading and trailing frames are not written.
  int halo;
  int Dy, Hy, Wy, d0, h0, w0, h_mode, w_mode;
  // x2 upsampled input (up2 = 1): Ho and Wo are the extents of the low-resolution
  // grid the tiles cover; y (and conv_out) is [N, Do, 2 Ho, 2 Wo, Cout] and the tile of
  // parity class cls writes output (2 h + cls / 2, 2 w + cls % 2)
  int up2;
  // e4m3 operands: the fp32 accumulator is multiplied by acc_scale (round to nearest)
  // before the first rounding to bf16; 1 otherwise
  float acc_scale;
};

// Implicit-GEMM convolution on tcgen05 (one CTA = R M-tiles x BN output channels).
struct ConvTCParams {
  EpiParams epi;
  int C;                   // channels of the NDHWC tensor the A tensor map reads
  int D, H, W;
  int KT, KR, KS;
  int st, sh, sw;
  int pt, ph, pw;          // leading pads (zero via TMA bounds, or reflect)
  int reflect_h, reflect_w;
  int tile_w, tile_h, R;   // M-tile = tile_h rows x tile_w pixels; R tiles per CTA
  int kc, n_chunks;        // channels per K chunk, chunks per tap
  int halo;                // 1: a stage holds one input-row halo for all KS taps
  int box_w;               // A box width in loaded elements
  int pitch_rows;          // shared-memory rows per A box (box_w rounded to 8)
  int a_tile_rows;         // rows between consecutive M-tiles in a stage
  int row_bytes;           // kc * 2
  int swz;                 // descriptor layout code (2 = 128B, 4 = 64B, 6 = 32B)
  int BN, n_sub, sub_n;    // CTA N = n_sub MMAs of sub_n columns
  int acc_stride;          // TMEM columns between M-tile accumulators
  int tmem_cols;
  int stages;
  uint32_t a_stage_bytes, b_stage_bytes, bar_off;
  uint32_t tx_bytes;       // bytes one stage's loads deliver
  int taps_per_stage;
  int stages_total;
  int k_splits, stages_per_split;
  int tiles_w, groups_h;
  int cp64;                // channel pitch of the packed weight
  int inject;              // test aid (see conv3d_tuning.inject)
  unsigned long long timeout_ns;
  float* partial;          // [k_splits][M][Cout] fp32 when k_splits > 1
  long long M_total;
};

// Channel-major implicit GEMM (persistent): D[channel][pixel] in TMEM, MMA
// M = 128 output channels, N = up to 256 output pixels of one tile.
struct ConvCMParams {
  EpiParams epi;
  int C;                   // channels of the NDHWC tensor the activation map reads
  int D, H, W;
  int KT, KR, KS;
  int st, sh, sw;
  int pt, ph, pw;
  int reflect_h, reflect_w;
  int tw, rh;              // pixel tile: rh output rows x tw output pixels
  int halo;                // 1: one run of tw + KS - 1 input pixels serves all KS taps
  int flat;                // 1 (with halo): H and W merged; a tile is tw consecutive
                           // positions of the flattened plane, row pitch W (needs
                           // stride 1, no W padding, zero H padding)
  int flat3;               // 1 (with flat): D, H and W merged; a tile is tw consecutive
                           // positions of the flattened volume and may span frames
                           // (needs stride 1 and no H / W padding; T zero padding reads
                           // positions outside the volume)
  int compact;             // 1 (with flat3): the flattened volume leaves out the KR - 1
                           // input rows below each frame's last output row, so a tile of
                           // tw positions covers output rows only; the activation map is
                           // an im2col map whose traversal runs over (W, Ho, Do)
  int tiles_d;             // output frames in the tile index (1 with flat3)
  int skip_pad;            // 1: tiles leave out the stages whose temporal tap reads only
                           // T padding
  int d_cheap;             // leading output frames whose tiles leave out all-padding
                           // temporal taps; the tile order puts them last (0 = plain order)
  int nbox;                // activation boxes per row of the tile (halo: 1..2, direct: 1)
  int rows_box;            // direct tiles: 1 = one box covers all rh rows (element
                           // stride sh along H), 0 = one box per row
  int box_w;               // loaded elements per activation box
  int run_pitch;           // shared-memory rows between the runs of consecutive output
                           // rows (also the tile's pixel pitch: valid columns are < tw)
  int N;                   // MMA N = round_up(rh * tw, 16)
  int kc, n_chunks, row_bytes;
  int taps_per_stage;
  int stages;
  uint32_t act_bytes, stage_bytes, bar_off, tx_bytes;
  uint32_t epi_off;        // per-warp [32][33] fp32 epilogue staging blocks
  int wgt_rows;            // weight box rows loaded per tap (<= 128; the MMA reads 128)
  int wgt_rows_last;       // the same for the last 128-channel tile (its own tensor map)
  uint32_t tx_bytes_last;  // bytes one stage of the last channel tile delivers
  uint32_t act_tx;         // activation bytes of one stage (part of both totals)
  int stages_total, k_splits, stages_per_split;
  int tiles_w, tiles_h, tiles_c;  // pixel tiles along W / H, 128-channel tiles
  int num_tiles;
  int acc_cols, nbuf, tmem_cols;
  int cp64;
  int inject;
  unsigned long long timeout_ns;
  float* partial;          // [k_splits][M][Cout] fp32 when k_splits > 1
  long long M_total;
  // fused L2 norm (k_splits == 1): the tiles_c channel tiles of a pixel tile run on
  // one CTA (tpu consecutive tiles per unit; tpu = 1 otherwise)
  int norm, tpu;
  int epi_groups;          // epilogue warpgroups (2 or 3): block = 128 + 128 * epi_groups
  // Pixel-major mode (Cout <= 128): the MMA takes the activations as A (M = 128 pixels
  // per half of the pixel tile) and the weights as B (N = pm_n = Cout rounded up to 16);
  // the accumulator of half h sits at column h * pm_cols, a thread of the epilogue owns
  // one pixel and needs no staging.
  int pm, pm_halves, pm_n, pm_cols;
  int wtap_rows;           // shared-memory weight rows per tap (128, or pm_n)
  int tma_store;           // output blocks on one output row (NCDHW: starting at a column
                           // that is a multiple of 8) are written by bulk
                           // tensor stores (y, value, conv maps) from the staging block
  uint32_t norm_off;       // shared den[N] (fp32) of the current pixel tile
  int norm_cs;             // channels per scratch row: Cout rounded up to 8
  uint16_t* vscratch;      // [grid][N][norm_cs] bf16 values, one slice per CTA
  // Paired last chunks (halo tiles, one split, Cin % 64 in 1..32): tap pairs
  // P = kt * KR + kr run in groups of two; a group is the full 64-channel chunks of
  // its first pair, then of its second, then one stage holding the last chunk of
  // both pairs as 32-channel, 64-byte rows (act: pair j at j * act_bytes / 2;
  // weights: pair j, tap s at (j * KS + s) * wtap_rows * 64).
  int pair, n_pairs;
  // Weight L2 prefetch: the weight producer asks L2 for the weight boxes of the stage
  // wpref stages ahead of the one it loads (0 = off).  Small layers read every weight
  // slice from HBM once, and two pipeline stages cannot hide that latency.
  int wpref;
  // Narrow-input gather mode (gather = 1; C = the real input channels, KR * KS * C <=
  // 32): one stage per temporal tap kt over tiles of one output row (rh = 1, direct
  // pixel order).  The activation map views the input as runs of 16-byte groups
  // (dims 8, W * C / 8 or W / 8, H, D, N or N * C); a stage's raw region (g_raw_off
  // past the operand rows) receives g_planes * KR rows of g_row_bytes; the expansion
  // turns them into 64-byte operand rows of K = g_K values.  The weights of every
  // (channel tile, kt) stay resident at g_wres_off, read once from g_wp.
  // x2 upsampled input (up2): the tiles run over the low-resolution grid once per
  // parity class (ncls = 4, class index next to the channel tile in the tile order);
  // class cls reads low-res row h + (-1, 0, 0)[r] (cls / 2 == 0) or h + (0, 0, 1)[r],
  // and its W taps are the run views shifted by (0, 1, 1) or (1, 1, 2) (cls % 2)
  int up2, ncls;
  int gather, g_K, g_cpp, g_planes, g_row_bytes;
  uint32_t g_raw_off, g_wres_off;
  const uint16_t* g_wp;     // packed weights [Cout][KT][KR][KS][cp64]
  // e4m3 operands (f8 = 1): C, kc, cp64 and every copy count two-byte channel pairs;
  // the MMA is kind::f8f6f4 (K = 32 one-byte channels per instruction, the same 32
  // bytes of each operand row as a bf16 K step) and epi.acc_scale scales the
  // accumulator
  int f8;
};

// Tensor maps of the paired last-chunk stages: 32-channel boxes, 64-byte swizzle.
struct CmHalfMaps {
  CUtensorMap act, wgt, wgt_last;
};

// Output tensor maps of the channel-major kernel's bulk-store epilogue (NDHWC,
// bf16, box = 32 channels x 32 pixels along W): y (for a haloed y, the view of the
// output inside it), value_out and conv_out (the last two repeat y when not
// requested), and the whole haloed y.
struct CmOutMaps {
  CUtensorMap y, val, conv;
  CUtensorMap yfull;  // haloed y: the whole tensor (halo rows that copy a block)
  CUtensorMap ycls[4];  // x2 upsampled input: y seen as the outputs of one parity class
};

}  // namespace vvc
