// Internal interface between the host API (fconv_api.cu) and the kernels
// (fconv_kernels.cu).  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fconv {

constexpr int kModeFused = 0;         // full epilogue, int8/bf16 output
constexpr int kModeAccumulators = 1;  // raw sums: int32 (int8 plans) / fp32 (bf16 plans)

// activation codes (the values of the public fconv_act)
constexpr int kActNone = 0, kActRelu = 1, kActLeakyRelu = 2, kActClippedRelu = 3, kActClamp = 4;

// Largest number of 64-wide k-blocks one fp32 accumulation may cover for
// int8 operands: 15 * 64 = 960 products of magnitude <= 2^14 stay below
// 2^24, so every partial sum is an exactly representable integer.
constexpr int kMaxExactKBlocks = 15;

// Everything the convolution kernel needs besides the B-operand tensor map.
struct ConvArgs {
  const void *a;       // activations NHWC, 16-bit (fp16 widened from int8, or bf16)
  const void *side;    // side input NHWC [M][K] (int8 or bf16), or nullptr
  const float *bias;   // [K]
  const float *scale_k;  // per-output-channel conv_input_scale [K], or nullptr (scalar)
  void *y;             // output [M][K] (int8/bf16, or int32/fp32 sums)
  int N, H, W, C, K, R, S, sh, sw, pt, pl, P, Q;
  long long M;         // N * P * Q
  int Ktot;            // R * S * C
  int num_kb;          // ceil(Ktot / 64)
  int kb_chunk;        // k-blocks per fp32 accumulation
  int num_n_tiles;     // ceil(K / BN)
  int num_tiles;       // ceil(M / 128) * num_n_tiles
  int b3d;             // tmap_b is the 3-D {64, rows, K / 64} view (K % 64 == 0)
  int kps;             // k-blocks a pipeline stage (1, or 2: TMA gather, unsplit,
                       // unchunked 128-pixel tiles of <= 128 channels); tmap_b's
                       // boxes are 64 * kps k-rows deep
  float conv_scale, side_scale;
  int act;             // kAct*
  // output pixel of GEMM row m (a phase of a strided transposed convolution
  // writes every o_sh-th row and o_sw-th column of an out_H x out_W output,
  // from (o_h0, o_w0)); omap == 0: row m is output pixel m
  int omap, out_H, out_W, o_sh, o_sw, o_h0, o_w0;
  float slope, lo, hi; // the activation as slope-then-clamp (see the epilogue)
  int use_side;
  int mode;
  int debug;
  unsigned long long timeout_ns;
  // split-K (TMA kernel): each tile's k-blocks in `splits` units of
  // kb_per_split; every unit writes its 32-bit partial sums (int32 for int8
  // plans, fp32 for bf16) to `partial`, and the last unit of a tile portion
  // to arrive (counted in `counters`, zeroed by the prep launch) adds them
  // in split order and runs the epilogue.  splits == 1: no partials.
  int splits, kb_per_split;
  uint32_t *partial;
  int *counters;
  // halo gather (stride 1, C == 64; Gather::kTmaHalo): a tile covers
  // halo_tr whole output rows of one image (tiles_per_img tiles an image);
  // its GEMM row i is the pixel (i / halo_q, i % halo_q) of those rows
  // padded to halo_q = Q + S - 1 columns, an output pixel when the column is
  // below Q, the row below halo_tr and the image row below P (the other
  // rows are computed and dropped).  The tile reads a window of halo_rows =
  // halo_tr + R - 1 input rows x halo_q pixels.  Shared memory: two
  // 16-bit windows of halo_slot bytes, two int8 stagings of halo_stg bytes
  // (int8 plans), then the resident filter tile.  w_i8: the caller's int8
  // filter, which int8 plans widen inside the kernel (no prep launch).
  int halo_q, halo_tr, halo_rows, tiles_per_img, halo_slot, halo_stg;
  const int8_t *w_i8;
  // two MMA issuers splitting each k-block's k16 steps into two
  // accumulators (TMA im2col, unsplit, 128-pixel tiles of <= 128 channels)
  int kdual;
};

// How the kernel gathers the A (activation) tile of each k-block.
enum class Gather {
  kCpAsync = 0,  // 16-byte cp.async per (pixel, 8 channels) with zero fill; any C % 8 == 0
  kTmaIm2col = 1, // one TMA im2col load of 128 pixels x 64 channels; needs C % 64 == 0
  // one tiled TMA load a tile of the input window its pixels read (stride
  // 1, C == 64), the filter tile resident; each tap's A is a row shift of
  // the window
  kTmaHalo = 2
};

// The halo gather's shared memory: two 16-bit input windows (1024-byte
// multiples), for int8 plans two stagings of the int8 window (512-byte
// multiples), and the resident filter tile (at most 9 k-blocks of 64 x 64),
// kHaloRegion bytes in all.
constexpr int kHaloRegion = 205 * 1024;
constexpr int kHaloBMax = 72 * 1024;

// m_sub: 128-pixel sub-tiles per output tile (1, or 2 on the TMA gather
// with block_n <= 128; args.num_tiles counts tiles of 128 * m_sub pixels).
// tmap_b: the filter as a [rows][K] 16-bit matrix (HWIO order, output
// channels contiguous), boxes of 64 x 64; with args.b3d the 3-D view
// {64 channels, rows, K / 64 blocks} with boxes of {64, 64, block_n / 64}.  overlap: the launch directly
// before this one on the stream is this run's prep launch, which the
// convolution may overlap (programmatic dependent launch).
// widen: int8 plans on the TMA gather, unsplit, block_n <= 128: tmap_a maps
// the int8 input itself (64-byte pixel rows) and the kernel widens it.
// Gather::kTmaHalo: tmap_a is the tiled map of the input itself (int8
// unswizzled, bf16 128-byte swizzled) with a {64, halo_q, halo_rows, 1}
// box; block_n 64, m_sub 1 or 2, unsplit, one fp32 accumulation, the grid
// a multiple of num_n_tiles (each CTA keeps one output-channel tile); int8:
// args.w_i8 is the caller's filter and tmap_b is unused (no prep launch).
cudaError_t launch_conv(int block_n, int m_sub, bool is_int8, Gather gather,
                        const CUtensorMap &tmap_a, const CUtensorMap &tmap_b,
                        const ConvArgs &args, int grid, bool overlap, cudaStream_t stream,
                        bool widen = false);
// Whether a gather mode has a kernel for this output-channel tile; chunked
// int8 sums on the cp.async path need a third TMEM region (BN <= 128).
bool gather_supports(Gather gather, int block_n, bool chunked, int m_sub = 1);
// Which input elements the prep launch copies (int8 widened to fp16, bf16
// as it is) into the [N][P][Q][C] copy the convolution reads.  Dense
// (mode 0, int8 only): all of x, P x Q = H x W.  Subsampled (1): for a 1x1
// filter with a stride above 1 the convolution reads only
// x[n, p*sh, q*sw, :], so only those pixels are copied, and the convolution
// reads the copy as a 1x1 stride-1 input.  Upsampled (2): a transposed
// convolution with stride (sh, sw) is the stride-1 one on x with sh-1 zero
// rows (sw-1 zero columns) inserted between its rows (columns): copy pixel
// (n, a, b) is x[n, a/sh, b/sw, :] when sh divides a and sw divides b, else
// zero; P = (H-1)*sh + 1, Q = (W-1)*sw + 1.
// Division by an invariant d >= 1 of any n < 2^31: q = (umulhi(n, m) + n) >> l
// with l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1 (the
// multiply-high method of Granlund and Montgomery, "Division by invariant
// integers using multiplication", 1994).
struct FastDiv {
  uint32_t d, m, l;
};
constexpr int kCopyDense = 0, kCopySubsample = 1, kCopyUpsample = 2;
struct WidenMap {
  int mode;
  int C, H, W, P, Q, sh, sw;
  FastDiv units_per_pixel, pq, q, div_sh, div_sw;   // filled in by launch_prep
  // filter copy: with tap_nR > 0 the copy is [tap_nR][tap_nS][C][K]
  // whose tap (j, l) is w[tap_r0 + tap_rstep*(tap_nR-1-j)][tap_s0 +
  // tap_sstep*(tap_nS-1-l)] of the caller's [tap_R][tap_S][C][K] filter
  // (flipped, and for a phase of a strided transposed convolution every
  // stride-th tap); tap_nR == 0 copies the filter as it is
  int tap_nR, tap_nS, tap_R, tap_S, tap_r0, tap_s0, tap_rstep, tap_sstep;
};
// Filter copy (w != nullptr: `rows` rows of K values into the 16-bit
// [rows][K] wt, int8 widened to fp16, rows mapped through the map's taps)
// and the input copy (n elements, a multiple of 16; int8 widened to fp16),
// in one launch (a second, tiny one when a dense n is not a multiple of 64).
// zero / zero_n: split-K counters the launch clears (nullptr, 0: none).
cudaError_t launch_prep(bool is_int8, const void *w, uint16_t *wt, int rows, int K,
                        const void *x, __half *xh, long long n, const WidenMap &map,
                        int *zero, int zero_n, int sm_count, cudaStream_t stream);
cudaError_t status_read_and_clear(cudaStream_t stream, unsigned int *out);
// Resource description of the kernel whose launch failed last on this thread.
const char *last_launch_note();

}  // namespace fconv
