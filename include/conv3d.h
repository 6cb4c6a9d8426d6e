/*
 * conv3d.h — C ABI of the GB300 (sm_103a) video-VAE convolution library.
 *
 * The library computes the bf16 forward convolution of a video VAE layer as
 * an implicit GEMM over channels-last activations, with an optional fused
 * post-operation epilogue, and a standalone form of that epilogue.
 *
 * Sources (web pages, cited by title and section):
 *  - ROCm/FlyDSL issue "[Feature]: conv3d_implicit — accept and emit NDHWC so
 *    chained convs skip the layout round-trip", section "Ask": the op
 *    conv3d_implicit(x, weight, bias, stride, padding, layout, out_layout) with
 *    NCDHW or NDHWC input and output; comment "The call site is already a clean
 *    drop-in": spatial reflect pad + temporal causal zero pad.
 *  - ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes to conv3d
 *    tests", sections "T=1 degeneration" and "Downsample Conv2d": rank-4
 *    (T=1) convolutions and the stride-2 downsample.
 *  - cuDNN frontend doc "Fused Conv3D + Bias + Residual + RMSNorm + SiLU",
 *    sections "Operation Contract" (epilogue arithmetic and its BF16 rounding
 *    points), "Requirements" (16-byte alignment, no overlap), "Weight Packing"
 *    (OITRS -> OTRSI, Ci padded to a multiple of 64), "Spatial Padding Variant"
 *    (zero bottom row and right column), "Standalone Normalization and Padding
 *    Variant" (post-operations without a convolution).
 *
 * Conventions for every entry point:
 *  - Tensor pointers are caller-owned DEVICE memory of the current CUDA
 *    device.  The library never allocates, never frees and never synchronises
 *    the stream (except conv3d_get_device_status, which reads a status word).
 *  - bf16 tensors are dense and contiguous in their declared layout, 16-byte
 *    aligned.  fp32 vectors (bias, residual_bias, gamma) hold Cout values and
 *    are 16-byte aligned.
 *  - Outputs and workspace must not overlap any operand or each other.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Every argument is validated before anything is launched; on a negative
 *    return nothing was enqueued.  A CUDA launch error returns
 *    CONV3D_ERR_CUDA.  A device-side wait that ran out of time records
 *    CONV3D_ERR_DEVICE_TIMEOUT in a device status word, read with
 *    conv3d_get_device_status.
 *  - Rank-4 (N, C, H, W) tensors are passed as D = 1 with KT = 1.
 */
#ifndef VVC_CONV3D_H
#define VVC_CONV3D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* conv3d_stream_t; /* same type as cudaStream_t */

/* ---- status codes ------------------------------------------------------------ */
enum {
  CONV3D_OK = 0,
  CONV3D_ERR_INVALID_ARG = -1,   /* null pointer, bad shape or flag combination */
  CONV3D_ERR_UNSUPPORTED = -2,   /* valid request outside what the kernels cover */
  CONV3D_ERR_MISALIGNED = -3,    /* a tensor pointer is not 16-byte aligned */
  CONV3D_ERR_OVERLAP = -4,       /* an output / workspace overlaps another buffer */
  CONV3D_ERR_WORKSPACE = -5,     /* workspace missing or too small */
  CONV3D_ERR_CUDA = -6,          /* a CUDA runtime / driver call failed */
  CONV3D_ERR_DEVICE_TIMEOUT = -7, /* a kernel's bounded wait ran out (device word) */
  CONV3D_ERR_SCRATCH_LIMIT = -8   /* conv3d_fwd_static_scratch: the call needs more scratch
                                     than the library's static 16 MiB buffer */
};

/* ---- layouts and padding ------------------------------------------------------ */
enum { CONV3D_NCDHW = 0, CONV3D_NDHWC = 1 };
enum { CONV3D_PAD_ZERO = 0, CONV3D_PAD_REFLECT = 1 };
enum { CONV3D_DTYPE_BF16 = 0, CONV3D_DTYPE_E4M3 = 1 };

/* Padding of one spatial dimension.  Zero: coordinates outside [0, L) read 0
 * (a causal temporal pad is before = 2, after = 0).  Reflect: PyTorch 'reflect'
 * (edge not repeated); needs before, after < L. */
typedef struct {
  int32_t before;
  int32_t after;
  int32_t mode;
} conv3d_pad;

/* ---- epilogue flags ([cuDNN page] "Operation Contract") --------------------------
 * With acc the fp32 accumulator and B() the fp32 -> bf16 round to nearest even:
 *   conv  = B(acc)
 *   main  = B(conv + bias[c])                        if CONV3D_EPI_BIAS, else conv
 *   skip  = residual, or B(residual + residual_bias[c]) with RESIDUAL_BIAS
 *   value = B(main + skip)                           if CONV3D_EPI_RESIDUAL, else main
 *   with CONV3D_EPI_L2NORM_SILU, over the full channel row of each pixel:
 *     den = max(sqrt(sum_c value_c^2), 1e-12); normalized = B(value / den)
 *     scaled = B(normalized * sqrt(Cout)); affine = B(scaled * gamma[c])
 *     y = B(affine / (1 + exp(-affine)))
 *   otherwise y = value.
 * No reassociation: every B() above is applied. */
enum {
  CONV3D_EPI_BIAS = 1,
  CONV3D_EPI_RESIDUAL = 2,
  CONV3D_EPI_RESIDUAL_BIAS = 4,   /* requires RESIDUAL */
  CONV3D_EPI_L2NORM_SILU = 8,     /* requires gamma */
  CONV3D_EPI_SAVE_VALUE = 16,     /* also write value (pre-normalisation) to value_out */
  CONV3D_EPI_OUT_PAD_BR = 32,     /* y gets a zero bottom row and right column:
                                     y spatial extent (Ho + 1, Wo + 1); not with L2NORM */
  CONV3D_EPI_PAD_CACHE = 64,      /* [cuDNN page] "Normalization and Padding Variant":
                                     requires L2NORM_SILU, NDHWC output, Cout % 8 == 0.
                                     y is the padded output [N, Do + 2, Ho + 2, Wo + 2,
                                     Cout]: the activations fill the interiors of planes
                                     2 .. Do + 1; every plane's one-pixel spatial border
                                     and the planes before the history_frames history
                                     planes are zeroed; the history planes' interiors
                                     are not written (the caller fills them).  cache_out
                                     [N, K, Ho, Wo, Cout], K = min(2, Do + history_frames):
                                     the last min(2, Do) activated frames go to its tail;
                                     its first K - min(2, Do) frames are not written. */
  CONV3D_EPI_DEBUG_STORE_CONV = 1 << 30 /* test aid: also write B(acc) to conv_out, NDHWC */
};

/* One convolution call.
 *  x          input, bf16 (or e4m3, see dtype), `layout`: NCDHW [N, Cin, D, H, W] or
 *             NDHWC [N, D, H, W, Cin].
 *  w_packed   weights packed by conv3d_pack_weight: [Cout][KT][KR][KS][Cin_pad64] bf16
 *             (e4m3: conv3d_pack_weight_e4m3).
 *  stride     (T, H, W) strides >= 1.
 *  pad        (T, H, W) paddings.  Output extent per dimension:
 *             (L + before + after - K) / stride + 1.
 *  y          output, bf16, `out_layout`, [N, Cout, Do, Ho, Wo] or [N, Do, Ho, Wo, Cout]
 *             (Ho + 1, Wo + 1 with CONV3D_EPI_OUT_PAD_BR; [N, Do + 2, Ho + 2, Wo + 2, Cout]
 *             with CONV3D_EPI_PAD_CACHE).
 *  bias, residual_bias, gamma   fp32 [Cout], as the flags require (else NULL).
 *  residual   bf16, `out_layout`, unpadded output shape (with CONV3D_EPI_RESIDUAL).
 *  value_out  bf16, `out_layout`, unpadded output shape (with CONV3D_EPI_SAVE_VALUE).
 *  conv_out   bf16 NDHWC unpadded output shape (with CONV3D_EPI_DEBUG_STORE_CONV).
 *  workspace  device scratch of at least conv3d_workspace_bytes() (may be NULL if 0).
 *  cache_out  bf16 NDHWC [N, min(2, Do + history_frames), Ho, Wo, Cout] (with
 *             CONV3D_EPI_PAD_CACHE, else ignored).
 *  history_frames   0, 1 or 2 activated frames the caller keeps in planes
 *             2 - history_frames .. 1 of y (with CONV3D_EPI_PAD_CACHE, else ignored).
 *  out_halo   (T, H, W) halo around the output inside y, so that the next call of a
 *             chain can read y as an already padded input and run a valid
 *             convolution (ROCm/FlyDSL issue "[Feature]: conv3d_implicit — ...",
 *             MiniMax-H3 comment: the causal temporal zero pad and the reflect
 *             spatial pad of every encoder convolution).  All zero: no halo, y is
 *             the plain output.  Otherwise y is NDHWC [N, Do + tb + ta, Ho + hb + ha,
 *             Wo + wb + wa, Cout] (tb = out_halo[0].before, ...), the output at
 *             offset (tb, hb, wb).  The T halo frames are never written (the caller
 *             keeps them, e.g. zeroed once for a causal chain); out_halo[0].mode must
 *             be CONV3D_PAD_ZERO.  H and W halos are at most 1 on a side and are
 *             written by every call: CONV3D_PAD_REFLECT fills them as PyTorch
 *             'reflect' padding of the output would (needs Ho, Wo >= 2),
 *             CONV3D_PAD_ZERO with zeros.  Requires NDHWC output, Cout % 8 == 0,
 *             and none of L2NORM_SILU, OUT_PAD_BR, PAD_CACHE.  residual, value_out
 *             and conv_out keep the unpadded output shape.
 *  input_upsample   0, or 2: the convolution reads the nearest-exact x2 upsampling of x
 *             along H and W (ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv
 *             shapes to conv3d tests", "Upsample Conv2d": the decoder's 3x3 convolution
 *             after nearest-exact x2), without writing the upsampled tensor: x is the
 *             low-resolution [N, D, H, W, Cin] (or NCDHW) tensor, and the convolution
 *             geometry (output extent, padding) applies to the [2H, 2W] upsampled grid.
 *             Requires KR = KS = 3, H and W stride 1 and zero padding (1, 1) along H and
 *             W (output [.., 2H, 2W]), NDHWC output, Cout % 8 == 0, and no RESIDUAL,
 *             L2NORM_SILU, SAVE_VALUE, OUT_PAD_BR, PAD_CACHE or out_halo.
 *  dtype      element type of x and w_packed: CONV3D_DTYPE_BF16 (0), or
 *             CONV3D_DTYPE_E4M3 (1): FP8 e4m3fn activations and weights with bf16
 *             output (ROCm/FlyDSL PR "[Flydsl] Add Qwen-Image VAE classic conv shapes
 *             to conv3d tests", "Summary" and "Test shapes": the FP8 suite feeds e4m3fn
 *             activations and weights, fp32 bias, and takes a bf16 output).  e4m3 x is
 *             NDHWC [N, D, H, W, Cin] bytes with Cin % 16 == 0; w_packed comes from
 *             conv3d_pack_weight_e4m3.  Products accumulate in fp32 as for bf16.  Not
 *             with input_upsample, the pixel-major kernel (conv3d_tuning.kernel = 1
 *             or 3, or Cout <= 16), or a narrow-input gather.
 *  fp8_scale  with CONV3D_DTYPE_E4M3: the accumulator is multiplied by fp8_scale
 *             (fp32, round to nearest) before the epilogue, conv = B(fp8_scale * acc),
 *             so per-tensor dequantisation scales of x and w enter as their product;
 *             must be finite and nonzero (1 for unscaled e4m3 values).  Ignored for
 *             bf16.  The pages give no scale convention; one per-tensor factor is the
 *             plainest that covers both unscaled and scaled e4m3 tensors. */
typedef struct {
  const void* x;
  int32_t layout;
  int32_t N, Cin, D, H, W;
  const void* w_packed;
  int32_t Cout, KT, KR, KS;
  int32_t stride[3];
  conv3d_pad pad[3];
  void* y;
  int32_t out_layout;
  uint32_t epi;
  const float* bias;
  const void* residual;
  const float* residual_bias;
  const float* gamma;
  void* value_out;
  void* conv_out;
  void* workspace;
  size_t workspace_bytes;
  void* cache_out;
  int32_t history_frames;
  conv3d_pad out_halo[3];
  int32_t input_upsample;
  int32_t dtype;
  float fp8_scale;
} conv3d_params;

/* Optional plan overrides (tests and tuning).  0 (or -1 where noted) = automatic. */
typedef struct {
  int32_t tile_w;      /* output pixels per M-tile row (<= 128) */
  int32_t tile_h;      /* output rows per M-tile (tile_w * tile_h <= 128) */
  int32_t R;           /* M-tiles per CTA */
  int32_t kc;          /* channels per K chunk: 16, 32 or 64 */
  int32_t BN;          /* output channels per CTA (multiple of 16) */
  int32_t halo;        /* 0 auto, 1 on, 2 off: one input-row halo serves all W taps */
  int32_t stages;      /* shared-memory pipeline depth */
  int32_t k_splits;    /* split of the reduction across CTAs (>= 1) */
  int32_t kernel;      /* 0 auto, 1 pixel-major kernel (M = pixels), 2 persistent kernel in
                          channel-major mode (M = 128 output channels, N = up to 256
                          pixels), 3 persistent kernel in pixel-major mode (M = 128 pixels
                          per half of the tile, N = Cout <= 128) */
  int32_t inject;      /* test aid: >0 makes the producer skip stage (inject-1) so a
                          bounded wait runs out; the call then reports a timeout */
  int32_t timeout_ms;  /* device wait limit (0 = default: 4000 ms, or the environment
                          variable CONV3D_TIMEOUT_MS when set) */
  int32_t im2col;      /* narrow inputs (Cin < 8): 0 auto, 1 gather the spatial taps into
                          a staged tensor first and run a (KT, 1, 1) convolution over it
                          (Cin * KR * KS <= 64), 2 neither, 3 gather the taps inside the
                          convolution kernel from TMA copies of the raw input rows
                          (Cin * KR * KS <= 32, W stride 1, W padding <= 1; not with
                          L2NORM_SILU).  Auto: 3 where it applies, else 1 where that
                          applies */
  int32_t pair;        /* 0 auto (= on), 1 on, 2 off: when the last 64-channel chunk of
                          the input holds at most 32 channels (Cin = 96, 160, ...) and
                          there are at least 2 (kt, kr) tap pairs, run the last chunks of
                          two consecutive tap pairs as one pipeline stage of 64-byte rows
                          instead of one half-empty stage each */
  int32_t prefetch;    /* weight L2 prefetch distance in pipeline stages: 0 auto (on for
                          layers whose CTAs run few tiles, so that every weight slice is a
                          first read from HBM), -1 off, > 0 that many stages ahead */
  int32_t compact;     /* 0 auto, 1 on, 2 off: tiles over the flattened volume (flat = 2
                          below) leave out the KR - 1 input rows under each frame's last
                          output row, so that every tile position is on an output row (the
                          activations then come through a TMA im2col map).  Auto: on when
                          that gives fewer tiles than both other flat forms */
} conv3d_tuning;

/* ---- weight packing ([cuDNN page] "Weight Packing") ------------------------------ */

/* Bytes of the packed weight: Cout * KT * KR * KS * round_up(Cin, 64) * 2. */
size_t conv3d_packed_weight_bytes(int32_t Cout, int32_t Cin, int32_t KT, int32_t KR,
                                  int32_t KS);

/* Packs checkpoint weights OITRS [Cout][Cin][KT][KR][KS] bf16 (device) into OTRSI
 * [Cout][KT][KR][KS][Cin_pad64] bf16 (device), zero-filling channels Cin..Cin_pad64-1.
 * Pack once; repack after the source weights change. */
int conv3d_pack_weight(const void* w_oitrs, int32_t Cout, int32_t Cin, int32_t KT,
                       int32_t KR, int32_t KS, void* w_packed, conv3d_stream_t stream);

/* FP8 e4m3fn weights (dtype CONV3D_DTYPE_E4M3): bytes of the packed weight,
 * Cout * KT * KR * KS * round_up(Cin, 128). */
size_t conv3d_packed_weight_bytes_e4m3(int32_t Cout, int32_t Cin, int32_t KT, int32_t KR,
                                       int32_t KS);

/* Packs e4m3fn OITRS [Cout][Cin][KT][KR][KS] bytes (device) into OTRSI
 * [Cout][KT][KR][KS][Cin_pad128] bytes (device), zero-filling channels
 * Cin..Cin_pad128-1 (the byte 0 is +0 in e4m3).  Same ownership and errors as
 * conv3d_pack_weight; both pointers 16-byte aligned and not overlapping. */
int conv3d_pack_weight_e4m3(const void* w_oitrs, int32_t Cout, int32_t Cin, int32_t KT,
                            int32_t KR, int32_t KS, void* w_packed, conv3d_stream_t stream);

/* ---- convolution ---------------------------------------------------------------- */

/* Scratch bytes conv3d_fwd needs for *p: the staged input (NCDHW input, Cin not a
 * multiple of 8, or the spatial im2col of a narrow input with its repacked weights),
 * split-reduction partial sums, and the bf16 value rows of the fused L2 norm.  0 when
 * none of these applies.  Returns a status; *bytes is set on success. */
int conv3d_workspace_bytes(const conv3d_params* p, size_t* bytes);
int conv3d_workspace_bytes_ex(const conv3d_params* p, const conv3d_tuning* tuning,
                              size_t* bytes);

/* Enqueues the convolution and its epilogue on `stream`. */
int conv3d_fwd(const conv3d_params* p, conv3d_stream_t stream);
int conv3d_fwd_ex(const conv3d_params* p, const conv3d_tuning* tuning,
                  conv3d_stream_t stream);

/* Allocation-free variant of conv3d_fwd (no counterpart on the source pages).
 * For callers that cannot allocate device memory when they run a convolution
 * (they only hold buffers handed to them, or allocation is forbidden in their
 * latency-critical or timed region): the scratch conv3d_fwd would take from
 * p->workspace (the channels-last staging copy of the input, the gathered taps
 * and repacked weights of a narrow input, split-reduction partial sums, the
 * fused norm's bf16 value rows, and the contiguous activations that the padded
 * output + cache places) comes from a static device array of 16 MiB that the
 * library module holds on every GPU it is loaded on, until the process exits.
 * p->workspace is ignored; inputs and outputs are the caller's as for conv3d_fwd.
 *  - A fused-norm call whose channel-major value rows do not fit runs on the
 *    pixel-major kernel, which needs none of them.  Other calls whose
 *    conv3d_workspace_bytes() exceeds 16 MiB return CONV3D_ERR_SCRATCH_LIMIT and
 *    launch nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture on the device.  The address is kept per device
 *    together with the CUDA context it was found in, and looked up again (also a
 *    first call, in this sense) when a device reset has replaced the context.
 *  - All calls share the one array per device and it keeps the last call's
 *    contents; every byte a call reads is written earlier in the same call, so
 *    nothing needs clearing.  Calls that can run at the same time on the GPU
 *    (different streams, or several host threads) race on the array: serialise
 *    them on one stream.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
int conv3d_fwd_static_scratch(const conv3d_params* p, conv3d_stream_t stream);

/* Number of kernel launches conv3d_fwd(_ex) enqueues for *p (for accounting). */
int conv3d_launch_count(const conv3d_params* p, const conv3d_tuning* tuning);

/* The plan conv3d_fwd_ex would run for *p (tests and tuning).  Host only: no
 * device work; the SM count comes from the current device (152 when there is
 * none).  Returns CONV3D_OK and fills *info, or the error the call would return
 * for an unsupported or invalid *p. */
typedef struct {
  int32_t kernel;           /* 1 pixel-major kernel (M = pixels), 2 channel-major
                               persistent kernel (M = output channels) */
  int32_t mma_n;            /* MMA N: pixels per tile (channel-major) or output
                               channels per tile (pixel-major) */
  int32_t stages_per_tile;  /* pipeline stages of one tile's whole reduction */
  int32_t k_splits;         /* split of the reduction across CTAs */
  int32_t paired;           /* 1: the last chunks of two tap pairs share a stage */
  int32_t im2col;           /* 1: the spatial taps are gathered into a staged tensor
                               before the conv, 2: inside the conv kernel */
  int32_t launches;         /* kernel launches of the call */
  int32_t grid;             /* CTAs of the convolution kernel */
  int32_t bulk_store;       /* 1: output blocks on one output row go out through bulk
                               tensor stores (channel-major kernel) */
  int32_t flat;             /* channel-major tiles: 0 rows of pixels, 1 runs of the
                               flattened H*W plane, 2 runs of the flattened D*H*W volume
                               (tiles span frames), 3 runs of the flattened volume of
                               output rows only (tiles span frames) */
} conv3d_plan_info;

int conv3d_plan(const conv3d_params* p, const conv3d_tuning* tuning, conv3d_plan_info* info);

/* ---- standalone post-operations ([cuDNN page] "Standalone Normalization and
 *      Padding Variant", contiguous output) ---------------------------------------
 * x: bf16 [rows][C] (rows = N*T*H*W, channels last).  main = B(x + input_bias) when
 * input_bias is non-NULL, else x; then the residual / L2-norm / SiLU steps of the
 * epilogue contract.  y: bf16 [rows][C].  value_out (optional, bf16 [rows][C])
 * receives the pre-normalisation value.  residual / residual_bias optional
 * (residual_bias requires residual). */
int l2norm_silu(const void* x, int64_t rows, int32_t C, const float* input_bias,
                const void* residual, const float* residual_bias, const float* gamma,
                void* y, void* value_out, conv3d_stream_t stream);

/* The same post-operations with padded output and cache ([cuDNN page] "Standalone
 * Normalization and Padding Variant").  x: bf16 NDHWC [N, T, H, W, C], C % 8 == 0.
 * previous: NULL, or the history_frames (1 or 2) prior activated frames, bf16
 * [N, history_frames, H, W, C].  padded_out: bf16 [N, T + 2, H + 2, W + 2, C]: the
 * frames [previous..., activated x...] end at plane T + 1 (history in planes
 * 2 - history_frames .. 1), zeros before them and on every plane's one-pixel
 * spatial border.  cache_out: bf16 [N, min(2, T + history_frames), H, W, C], the
 * last frames of that sequence.  value_out (optional): the pre-normalisation value,
 * [N, T, H, W, C].  input_bias, residual, residual_bias as in l2norm_silu.  All
 * pointers 16-byte aligned; outputs must not overlap each other or any input.
 * Two launches on `stream`; nothing is allocated. */
int l2norm_silu_pad(const void* x, int32_t N, int32_t T, int32_t H, int32_t W, int32_t C,
                    const float* input_bias, const void* residual, const float* residual_bias,
                    const float* gamma, const void* previous, int32_t history_frames,
                    void* padded_out, void* cache_out, void* value_out,
                    conv3d_stream_t stream);

/* ---- streaming causal convolution: input packing ([cuDNN page] "Causal Conv3D with
 *      Cache", and the "CausalConv3dWithCacheSm100" row of the API table: input/history
 *      packing with padding, then the convolution without bias) -------------------------
 * Builds the padded channels-last input of one chunk of a causal 3x3x3 convolution and
 * the raw history for the next chunk.
 * x: the chunk, bf16 [N, C, T, H, W] (NCTHW) at non-negative element strides
 *    x_strides[5] = (n, c, t, h, w); any view of device memory, 2-byte aligned.
 * previous: raw history frames, bf16 [N, history_frames, H, W, C] contiguous, 8-byte
 *    aligned; NULL exactly when history_frames = 0 (0, 1 or 2).
 * padded: bf16 [N, T + 2, H + 2, W + 2, Cp] contiguous (Cp >= C, Cp % 8 == 0, Cp <= 256;
 *    12 -> 16 on the page): planes 0 and 1 are the two frames before the chunk (history
 *    frames, a zero plane for each missing one: the causal padding), planes 2 .. T + 1
 *    the chunk; a one-pixel zero border in H and W; channels C .. Cp - 1 zero.
 * cache_out: bf16 [N, min(2, T + history_frames), H, W, C] contiguous, the last frames of
 *    [history..., chunk...] in order: the next chunk's previous.
 * padded and cache_out 16-byte aligned, overlapping neither each other nor an input.
 * The chunk's output is then conv3d_fwd over padded: NDHWC, Cin = Cp, valid padding,
 * weights packed by conv3d_pack_weight from [Cout, C, 3, 3, 3] (the packed layout pads
 * input channels to 64 with zeros, so it serves Cin = Cp as well).  One launch on
 * `stream`; nothing is allocated. */
int conv3d_causal_pack(const void* x, const int64_t* x_strides, int32_t N, int32_t C, int32_t T,
                       int32_t H, int32_t W, const void* previous, int32_t history_frames,
                       void* padded, int32_t Cp, void* cache_out, conv3d_stream_t stream);

/* ---- channels-last GroupNorm (+ SiLU) ([FlyDSL issue] MiniMax-H3 comment, "An extra
 *      argument for NDHWC": the GroupNorm between the encoder's convolutions, with
 *      time-isolated groups) ------------------------------------------------------------
 * x, y: bf16 NDHWC [N, D, H, W, C], C % 8 == 0, 8 <= C <= 2048; groups divides C and a
 * group is C / groups contiguous channels.  Statistics per (n, d, group) over
 * H * W * C / groups elements when time_isolated (each frame on its own), else per
 * (n, group) over D * H * W * C / groups: mean and biased variance, accumulated in fp32
 * per block and combined in fp64.  y = B((x - mean) / sqrt(var + eps) * gamma[c] +
 * beta[c]), then with silu y = B(y / (1 + exp(-y))).  gamma, beta: fp32 [C], or NULL for
 * 1 and 0.  workspace: at least group_norm_workspace_bytes() bytes of device memory.
 * All pointers 16-byte aligned; y must not overlap x, gamma, beta or the workspace.
 * Two launches on `stream`; nothing is allocated. */
size_t group_norm_workspace_bytes(int32_t N, int32_t D, int32_t H, int32_t W, int32_t C,
                                  int32_t groups, int32_t time_isolated);
int group_norm_silu(const void* x, int32_t N, int32_t D, int32_t H, int32_t W, int32_t C,
                    int32_t groups, int32_t time_isolated, float eps, const float* gamma,
                    const float* beta, int32_t silu, void* y, void* workspace,
                    size_t workspace_bytes, conv3d_stream_t stream);

/* ---- status ---------------------------------------------------------------------- */

/* Synchronises `stream`, then reads and clears the device status word: *status
 * is CONV3D_OK or CONV3D_ERR_DEVICE_TIMEOUT.  Returns CONV3D_ERR_CUDA if the copy
 * fails. */
int conv3d_get_device_status(int32_t* status, conv3d_stream_t stream);

const char* conv3d_status_string(int status);

/* Library ABI version (major * 100 + minor).  2.00: conv3d_params gained cache_out and
 * history_frames, conv3d_tuning gained pair; conv3d_plan, l2norm_silu_pad and the GroupNorm
 * calls were added.  3.00: conv3d_params gained out_halo and input_upsample.  3.10:
 * conv3d_params gained dtype and fp8_scale; conv3d_pack_weight_e4m3 and
 * conv3d_packed_weight_bytes_e4m3 were added.  3.20: conv3d_tuning gained compact;
 * conv3d_causal_pack was added. */
int conv3d_version(void);

/* sizeof() of the ABI structs, for bindings to check their mirrors:
 * which = 0 conv3d_params, 1 conv3d_tuning, 2 conv3d_pad, 3 conv3d_plan_info;
 * 0 otherwise. */
size_t conv3d_struct_size(int which);

#ifdef __cplusplus
}
#endif

#endif /* VVC_CONV3D_H */
