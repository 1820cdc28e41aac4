// Kernels of the fused Conv2D forward pass for sm_103a.
//
// The convolution is an implicit GEMM (the im2col view of
// "conv_grad_filter_ops.cc", Im2col, without materialising the patch
// matrix):
//     D[m][n] = sum_k A[m][k] * B[n][k]
//     m = (n_img, p, q) output pixel, n = output channel,
//     k = (r, s, c) in the HWIO flattening order,
//     A[m][k] = x[n_img, p*sh + r - pt, q*sw + s - pl, c] or 0 off the image,
//     B[n][k] = w[r, s, c, n].
// D accumulates in fp32 in tensor memory (TMEM) on the 5th-generation tensor
// cores (tcgen05.mma kind::f16).  sm_103a has no integer tensor-core MMA, so
// int8 operands are widened to fp16, where every int8 value is exact; each
// product is then at most 2^14 and exact in fp32, and the plan limits one
// fp32 accumulation to 960 k-values (15 k-blocks of 64), so every partial
// sum stays below 2^24 and is exact.  Longer reductions are split into such
// chunks and the chunks are summed in int32 by the epilogue, which makes the
// int8 result the exact int32 sum the TensorFlow kernel describes.
//
// CTA layout (288 threads, one CTA per SM, persistent over output tiles):
//   warps 0-3  loaders.  When C % 64 == 0, thread 0 alone loads each
//              k-block with two TMA copies: the 128 x 64 A tile by an im2col
//              load (the hardware walks the output pixels and zero-fills
//              padding taps) and the BN x 64 B tile by a tiled load.
//              Otherwise all 128 threads gather the A tile with 16-byte
//              cp.async (zero fill for padding taps) into the same
//              128-byte-swizzled K-major layout and thread 0 loads B by TMA.
//   warp 4     allocates TMEM; lane 0 issues the MMAs (4 per k-block).
//   warps 5-8  epilogue (warp w reads TMEM lanes 32*(w%4) .. +31): TMEM -> registers, BiasActivationOutputKernel's
//              three fp32 steps, rounding, saturation, 16-byte stores.
// The accumulator is double-buffered in TMEM so the epilogue of one tile
// overlaps the mainloop of the next.
#include <atomic>
#include <cstdio>

#include <utility>

#include "fconv_device.cuh"
#include "fconv_internal.h"

namespace fconv {

constexpr int kBM = 128;                // output pixels per tile (MMA M)
constexpr int kBK = 64;                 // k-values per k-block (128 bytes of 16-bit)
constexpr int kThreads = 288;
constexpr int kLoaderThreads = 128;
constexpr int kMmaWarp = 4;

template <int BN>
struct Cfg {
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages0 = (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
  // k-blocks of cp.async each loader keeps in flight beyond the newest one:
  // all stages but two (one being consumed by the MMA, one being refilled)
  static constexpr int kLag = kStages - 2;
  static constexpr bool kCanChunk = 3 * BN <= 512;
  static constexpr int kColsNeeded = kCanChunk ? 3 * BN : 2 * BN;
  static constexpr int kTmemCols = kColsNeeded <= 32    ? 32
                                   : kColsNeeded <= 64  ? 64
                                   : kColsNeeded <= 128 ? 128
                                   : kColsNeeded <= 256 ? 256
                                                        : 512;
  static constexpr int kBarOffset = kStages * kStageBytes;
  // after the barriers: each of the 4 epilogue warps' copy of the tile's
  // bias and per-channel scale ([warp][bias | scale][BN] floats), then its
  // output staging buffer (32 rows x 64 bytes)
  static constexpr int kParamOffset = kBarOffset + 256;
  static constexpr int kParamBytes = 4 * 2 * BN * 4;
  static constexpr int kOutOffset = kParamOffset + kParamBytes;
  static constexpr int kOutWarpBytes = 32 * 64;
  static constexpr int kSmemBytes = 1024 + kOutOffset + 4 * kOutWarpBytes;
  static_assert(kSmemBytes <= 232448, "dynamic shared memory per block");
  static_assert(kLag >= 2, "pipeline too shallow");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "MMA N in whole 64-channel B boxes");
};

struct Smem {
  uint64_t full_a[8];
  uint64_t full_b[8];
  uint64_t empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// The B (filter) tile of k-block kb and output-channel tile n_tile, MN-major:
// the filter is read as the [R*S*C][K] matrix of its HWIO layout (output
// channels contiguous), as BN / 64 blocks of 64 channels x 64 k-rows, each
// 8 KB, 128-byte swizzled (see sw128_mnmajor_desc).  Rows past R*S*C and
// channels past K read as zero.  b3d (K a multiple of 64): the tensor map
// views the matrix as {64 channels, rows, K / 64 channel blocks} and one
// copy of a {64, 64, BN / 64} box writes the whole tile in that layout;
// otherwise each block is its own 2-D copy.  The copies a producer issues,
// not their bytes, bound how fast it fills stages, so one copy is cheaper.
// KPS k-blocks a stage: the boxes are 64 * KPS k-rows deep, so each block of
// 64 channels holds the stage's KPS k-blocks one after another (8 KB each)
// and the blocks are 8 KB * KPS apart.
constexpr uint64_t kBStepK = 2048 >> 4;   // descriptor step of 16 k-rows
template <int BN, int KPS = 1>
__device__ __forceinline__ void load_b_tile(uint32_t dst, const CUtensorMap *map, int kb,
                                            int n_tile, int b3d, uint32_t bar) {
  if (b3d) {
    tma_load_3d(dst, map, 0, kb * kBK, n_tile * (BN / 64), bar);
  } else {
#pragma unroll
    for (int j = 0; j < BN / 64; ++j)
      tma_load_2d(dst + j * 8192 * KPS, map, n_tile * BN + 64 * j, kb * kBK, bar);
  }
}

// Four int8 values (one 32-bit word) to two fp16x2 words, exactly: with the
// sign bit flipped a byte b is u = b + 128 in [0, 255]; the fp16 bit pattern
// 0x6400 | u is 1024 + u, and subtracting 1152 (0x6480) leaves b.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(u, 0x64646464u, 0x4140);   // [u0, 0x64, u1, 0x64]
  const uint32_t b = __byte_perm(u, 0x64646464u, 0x4342);   // [u2, 0x64, u3, 0x64]
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
  lo = *reinterpret_cast<const uint32_t *>(&ha);
  hi = *reinterpret_cast<const uint32_t *>(&hb);
}

// Widen int8 pixel rows [p0, p1) of a staged window (64 bytes a pixel) into
// the 16-bit window the MMA reads (128 bytes a pixel, 128-byte swizzle:
// 16-byte chunk j of row r at j ^ (r & 7), as a TMA copy writes it), by one
// warp: four 16-byte pieces of each lane in flight before their stores.
__device__ __forceinline__ void widen_rows(const uint8_t *src, uint8_t *dst, int p0, int p1) {
  const int lane = threadIdx.x & 31;
  const int n = (p1 - p0) * 4;   // 16-byte pieces
  const uint8_t *s0 = src + p0 * 64;
  for (int i0 = 0; i0 < n; i0 += 128) {
    uint4 in[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int i = i0 + g * 32 + lane;
      if (i < n) in[g] = *reinterpret_cast<const uint4 *>(s0 + i * 16);
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int i = i0 + g * 32 + lane;
      if (i < n) {
        const int r = p0 + (i >> 2), pc = i & 3;
        uint4 lo, hi;
        i8x4_to_f16x4(in[g].x, lo.x, lo.y);
        i8x4_to_f16x4(in[g].y, lo.z, lo.w);
        i8x4_to_f16x4(in[g].z, hi.x, hi.y);
        i8x4_to_f16x4(in[g].w, hi.z, hi.w);
        uint8_t *row = dst + r * 128;
        *reinterpret_cast<uint4 *>(row + (((2 * pc) ^ (r & 7)) << 4)) = lo;
        *reinterpret_cast<uint4 *>(row + (((2 * pc + 1) ^ (r & 7)) << 4)) = hi;
      }
    }
  }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
  return __uint_as_float(b16 << 16);
}

// Raw int32 sums of one 32-column slice (chunked int8 accumulation).
__device__ __forceinline__ void store_i32_slice(const ConvArgs &a, long long m, int col0,
                                                const uint32_t (&u)[32]) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int col = col0 + 4 * g;
    if (col < a.K)
      stg_v4(static_cast<uint32_t *>(a.y) + m * a.K + col,
             make_uint4(u[4 * g], u[4 * g + 1], u[4 * g + 2], u[4 * g + 3]));
  }
}

// One 32-column slice of the epilogue for one output row, streamed in
// groups of 16 (int8) or 8 (bf16) columns so few values are live at once.
// vals: the 32 pre-epilogue sums as fp32 (exact integers for int8 plans).
// Columns at or beyond K are skipped (K is a multiple of the group width).
// The activation on the fp32 value after the bias add, branch-free: a
// slope for negative values (one rounding; 1 is exact), then a clamp to
// [lo, hi] (infinite bounds are exact).  The host sets slope, lo and hi:
// none (1, -inf, inf), Relu (1, 0, inf), leaky (alpha, -inf, inf), clipped
// (1, 0, alpha), clamp (1, alpha, beta).  For v < 0 the first line is
// round(v * slope) + 0, for v >= 0 it is 0 * slope + v: the same value as
// "v < 0 ? v * slope : v".
__device__ __forceinline__ float activation(float v, const ConvArgs &a) {
  v = __fadd_rn(__fmul_rn(fminf(v, 0.0f), a.slope), fmaxf(v, 0.0f));
  return fminf(fmaxf(v, a.lo), a.hi);
}

// Output pixel (flat [N][out_H][out_W] index) of GEMM row m.
__device__ __forceinline__ long long out_pixel(const ConvArgs &a, long long m) {
  if (!a.omap) return m;
  const long long PQ = static_cast<long long>(a.P) * a.Q;
  const long long n = m / PQ;
  const int rem = static_cast<int>(m - n * PQ);
  const int p = rem / a.Q, q = rem - p * a.Q;
  return (n * a.out_H + a.o_h0 + static_cast<long long>(p) * a.o_sh) * a.out_W + a.o_w0 +
         static_cast<long long>(q) * a.o_sw;
}

// 16-byte groups of a 32-column slice (of outputs, or of side-input words):
// int8 2 x 16 columns, bf16 4 x 8.
template <bool IS_INT8>
struct SliceGroups {
  static constexpr int kGroups = IS_INT8 ? 2 : 4;
  static constexpr int kCols = IS_INT8 ? 16 : 8;   // columns per group
};

template <bool IS_INT8>
__device__ __forceinline__ void load_side_words(const ConvArgs &a, long long m, int col0,
                                                uint4 *words) {
#pragma unroll
  for (int h = 0; h < SliceGroups<IS_INT8>::kGroups; ++h) {
    const int col = col0 + h * SliceGroups<IS_INT8>::kCols;
    words[h] = (a.use_side && col < a.K)
                   ? ldg_nc_v4(static_cast<const uint8_t *>(a.side) +
                               (m * a.K + col) * (IS_INT8 ? 1 : 2))
                   : make_uint4(0, 0, 0, 0);
  }
}

// The fused epilogue of one 32-column slice of one output row, in the order
// of BiasActivationOutputKernel: (1) scale, (2) side input (one fused
// rounding), (3) bias, then the activation and the output rounding.  Each
// step runs over 16 columns before the next, so 16 independent chains
// interleave (two halves a slice keep the registers in bounds).  The
// explicit round-to-nearest intrinsics keep nvcc from contracting (1) and
// (3) into an fma.  vals: the 32 sums as fp32 (exact integers for int8
// plans); sv: the slice's side-input words (int8 2 x 16 bytes, bf16 4 x 8
// values); bias_p / scale_p: the slice's first column (scale_p read only
// with a per-channel scale).  out: the slice packed as it is stored (int8
// 2 x 16 codes, bf16 4 x 8 values).  GENERAL_ACT: the slope-then-clamp
// activation; otherwise (no activation or Relu) only the lower bound a.lo
// (-inf or 0).
template <bool IS_INT8, bool GENERAL_ACT>
__device__ __forceinline__ void fused_slice(const ConvArgs &a, const float (&vals)[32],
                                            const uint4 (&sv)[SliceGroups<IS_INT8>::kGroups],
                                            const float *bias_p, const float *scale_p,
                                            uint4 (&out)[SliceGroups<IS_INT8>::kGroups]) {
  uint32_t sw[SliceGroups<IS_INT8>::kGroups * 4];
#pragma unroll
  for (int g = 0; g < SliceGroups<IS_INT8>::kGroups; ++g) {
    sw[4 * g + 0] = sv[g].x; sw[4 * g + 1] = sv[g].y;
    sw[4 * g + 2] = sv[g].z; sw[4 * g + 3] = sv[g].w;
  }
  uint32_t wd[IS_INT8 ? 8 : 16];   // the packed outputs
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c0 = 16 * h;
    float v[16];
    if (a.scale_k) {   // (1) per output channel: every lane reads the same 16 bytes
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 s4 = *reinterpret_cast<const float4 *>(scale_p + c0 + 4 * q);
        v[4 * q + 0] = __fmul_rn(vals[c0 + 4 * q + 0], s4.x);
        v[4 * q + 1] = __fmul_rn(vals[c0 + 4 * q + 1], s4.y);
        v[4 * q + 2] = __fmul_rn(vals[c0 + 4 * q + 2], s4.z);
        v[4 * q + 3] = __fmul_rn(vals[c0 + 4 * q + 3], s4.w);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(vals[c0 + i], a.conv_scale);
    }
    if (a.use_side) {   // (2)
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int c = c0 + i;
        float sd;
        if (IS_INT8) {
          // byte b in offset binary as the mantissa of 2^23 is the float
          // 2^23 + b + 128; subtracting 2^23 + 128 leaves b exactly
          sd = __fsub_rn(__uint_as_float(__byte_perm(sw[c / 4] ^ 0x80808080u, 0x4B000000u,
                                                     0x7540u + (c % 4))),
                         8388736.0f);
        } else {
          sd = bf16_bits_to_float((sw[c / 2] >> (16 * (c % 2))) & 0xFFFFu);
        }
        v[i] = __fmaf_rn(sd, a.side_scale, v[i]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {   // (3) every lane reads the same 16 bytes
      const float4 b4 = *reinterpret_cast<const float4 *>(bias_p + c0 + 4 * q);
      v[4 * q + 0] = __fadd_rn(v[4 * q + 0], b4.x);
      v[4 * q + 1] = __fadd_rn(v[4 * q + 1], b4.y);
      v[4 * q + 2] = __fadd_rn(v[4 * q + 2], b4.z);
      v[4 * q + 3] = __fadd_rn(v[4 * q + 3], b4.w);
    }
    if (IS_INT8) {
      // The clamp to [lo, 127] before rounding: the activation's lower
      // bound (Relu 0, none -inf) merged with the int8 range.  Saturating
      // after a round-half-even gives the same code as rounding the clamped
      // value.
      const float lo = GENERAL_ACT ? -128.0f : fmaxf(a.lo, -128.0f);
      uint32_t t[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        float x = GENERAL_ACT ? activation(v[i], a) : v[i];
        x = fminf(fmaxf(x, lo), 127.0f);
        // 1.5 * 2^23 + x, x in [-128, 127]: the fp32 ulp there is 1, so the
        // add rounds x half to even and the low byte of the sum's bits is
        // that integer in two's complement
        t[i] = __float_as_uint(__fadd_rn(x, 12582912.0f));
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        wd[4 * h + k] = __byte_perm(__byte_perm(t[4 * k], t[4 * k + 1], 0x0040u),
                                    __byte_perm(t[4 * k + 2], t[4 * k + 3], 0x0040u), 0x5410u);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float r0 = GENERAL_ACT ? activation(v[2 * k], a) : fmaxf(v[2 * k], a.lo);
        const float r1 = GENERAL_ACT ? activation(v[2 * k + 1], a) : fmaxf(v[2 * k + 1], a.lo);
        // both round to nearest even in one conversion; .x is the low half
        const __nv_bfloat162 pr = __floats2bfloat162_rn(r0, r1);
        wd[8 * h + k] = *reinterpret_cast<const uint32_t *>(&pr);
      }
    }
  }
#pragma unroll
  for (int g = 0; g < SliceGroups<IS_INT8>::kGroups; ++g)
    out[g] = make_uint4(wd[4 * g], wd[4 * g + 1], wd[4 * g + 2], wd[4 * g + 3]);
}

// Raw sums of one 32-column slice of row m (the accumulator-only mode):
// int32 for int8 plans, fp32 for bf16 plans; 4 columns per store.
template <bool IS_INT8>
__device__ __forceinline__ void store_raw_slice(const ConvArgs &a, long long m, int col0,
                                                const float (&vals)[32]) {
  const int K = a.K;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int col = col0 + 4 * g;
    if (col < K) {
      uint4 o;
      if (IS_INT8) {
        o.x = static_cast<uint32_t>(__float2int_rn(vals[4 * g + 0]));
        o.y = static_cast<uint32_t>(__float2int_rn(vals[4 * g + 1]));
        o.z = static_cast<uint32_t>(__float2int_rn(vals[4 * g + 2]));
        o.w = static_cast<uint32_t>(__float2int_rn(vals[4 * g + 3]));
      } else {
        o.x = __float_as_uint(vals[4 * g + 0]);
        o.y = __float_as_uint(vals[4 * g + 1]);
        o.z = __float_as_uint(vals[4 * g + 2]);
        o.w = __float_as_uint(vals[4 * g + 3]);
      }
      stg_v4(static_cast<uint32_t *>(a.y) + m * K + col, o);
    }
  }
}

// The fused epilogue of one 32-column slice for a whole warp (all 32 lanes
// call it; lane l holds row l), with the stores coalesced: the rows'
// 16-byte groups pass through the warp's shared-memory buffer `stage` (32
// rows x kGroups x 16 bytes) so that each store instruction writes whole
// 32-byte row segments of consecutive lanes (kGroups lanes per row).
// Groups sit in the buffer rotated by the row's position within its
// eight-row bank window, so neither the writes nor the reads conflict.
// mo / valid: this lane's output pixel and whether its row exists.
// side_pre: the slice's side words loaded ahead (load_side_words), or
// nullptr to load them here (valid rows only).  bias_c / scale_c: the
// slice's 32 bias and per-channel scale values in shared memory (scale_c
// nullptr: the scalar a.conv_scale).  st_mo / st_ok: output pixel and
// existence of the row this lane stores in store round k (row
// (32 k + lane) / kGroups), from coalesced_rows.
template <bool IS_INT8, bool GENERAL_ACT>
__device__ __forceinline__ void epilogue_slice_coalesced(const ConvArgs &a, long long mo,
                                                         bool valid, int col0,
                                                         const float (&vals)[32],
                                                         const uint4 *side_pre,
                                                         const float *bias_c,
                                                         const float *scale_c, uint4 *stage,
                                                         const long long *st_mo,
                                                         const bool *st_ok) {
  using G = SliceGroups<IS_INT8>;
  constexpr int kG = G::kGroups;
  constexpr int elt = IS_INT8 ? 1 : 2;
  const int lane = threadIdx.x & 31;
  const int K = a.K;
  const float *scale_p = scale_c ? scale_c : a.scale_k + col0;
  // swizzle of row r: 8 / kG consecutive rows share a 128-byte bank window
  auto swz = [](int r) { return (r / (8 / kG)) % kG; };
  uint4 sv[kG], outw[kG];
#pragma unroll
  for (int gi = 0; gi < kG; ++gi) {
    sv[gi] = make_uint4(0, 0, 0, 0);
    if (side_pre) sv[gi] = side_pre[gi];
    else if (a.use_side && valid && col0 + G::kCols * gi < K)
      sv[gi] = ldg_nc_v4(static_cast<const uint8_t *>(a.side) +
                         (mo * K + col0 + G::kCols * gi) * elt);
  }
  fused_slice<IS_INT8, GENERAL_ACT>(a, vals, sv, bias_c, scale_p, outw);
#pragma unroll
  for (int gi = 0; gi < kG; ++gi) stage[lane * kG + (gi ^ swz(lane))] = outw[gi];
  __syncwarp();
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const int piece = k * 32 + lane;
    const int r = piece / kG, q = piece % kG;   // row and group this lane stores
    const uint4 v = stage[r * kG + (q ^ swz(r))];
    const int col = col0 + G::kCols * q;
    if (st_ok[k] && col < K) stg_v4(static_cast<uint8_t *>(a.y) + (st_mo[k] * K + col) * elt, v);
  }
  __syncwarp();   // the buffer is free for the next slice
}

// The rows a lane stores in the coalesced rounds: round k stores row
// (32 k + lane) / kGroups, whose output pixel and existence its own lane
// holds.  The whole warp calls this, once per tile.
template <bool IS_INT8>
__device__ __forceinline__ void coalesced_rows(long long mo, bool valid, long long *st_mo,
                                               bool *st_ok) {
  constexpr int kG = SliceGroups<IS_INT8>::kGroups;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const int r = (k * 32 + lane) / kG;
    st_mo[k] = __shfl_sync(0xffffffffu, mo, r);
    st_ok[k] = __shfl_sync(0xffffffffu, static_cast<int>(valid), r) != 0;
  }
}

template <bool IS_INT8>
__device__ __forceinline__ void epilogue_slice_warp(const ConvArgs &a, long long mo, bool valid,
                                                    int col0, const float (&vals)[32],
                                                    const uint4 *side_pre, const float *bias_c,
                                                    const float *scale_c, uint4 *stage,
                                                    const long long *st_mo, const bool *st_ok) {
  if (a.act > kActRelu)
    epilogue_slice_coalesced<IS_INT8, true>(a, mo, valid, col0, vals, side_pre, bias_c, scale_c,
                                            stage, st_mo, st_ok);
  else
    epilogue_slice_coalesced<IS_INT8, false>(a, mo, valid, col0, vals, side_pre, bias_c, scale_c,
                                             stage, st_mo, st_ok);
}

// General path: cp.async gather of A by 4 loader warps, 4 epilogue warps.
// int8 sums longer than one exact chunk are folded into int32 in a third
// TMEM region, so chunked plans use BN <= 128.
template <int BN, bool IS_INT8>
__global__ void __launch_bounds__(kThreads, 1)
    conv_fprop_cpasync_kernel(const __grid_constant__ CUtensorMap tmap_b, const ConvArgs args) {
  using C = Cfg<BN>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kIdesc = idesc_f16(kBM, BN, !IS_INT8, /*b_mn=*/true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kStages * C::kABytes;
  Smem *bars = reinterpret_cast<Smem *>(smem + C::kBarOffset);
  volatile int *abort_flag = &bars->abort_flag;

  // taken from lane 0 so that the compiler sees a warp-uniform value and the
  // role branches below are uniform
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->full_a[s]), kLoaderThreads);
      mbar_init(smem_u32(&bars->full_b[s]), 1);
      mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->acc_full[s]), 1);
      mbar_init(smem_u32(&bars->acc_empty[s]), 4);
    }
    mbar_init(smem_u32(&bars->mma_done), 1);
    bars->abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = __shfl_sync(0xffffffffu, bars->tmem_base, 0);

  const int num_kb = args.num_kb;
  const int kb_chunk = args.kb_chunk;
  const int n_chunks = (num_kb + kb_chunk - 1) / kb_chunk;

  if (warp < 4) {
    // ------------------------------------------------------------ loaders
    const int t = threadIdx.x;
    const int j = t & 7;            // 16-byte chunk (8 channels) of the 128-byte row
    const int rsub = t >> 3;        // rows rsub + 16*i, i = 0..7
    const int Cc = args.C, Hh = args.H, Ww = args.W, Rr = args.R, Ss = args.S;
    const long long PQ = static_cast<long long>(args.P) * args.Q;
    const uint16_t *act = static_cast<const uint16_t *>(args.a);
    uint32_t stage = 0, phase = 0, arr_stage = 0;
    uint32_t issued = 0;            // TMA issues by thread 0
    int pending = 0;
    bool ok = true;
    const bool drop = (args.debug & 1) != 0;
    griddep_wait();   // the widened input and filter copy of the prep launch

    for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
      const int m_tile = tile / args.num_n_tiles;
      const int n_tile = tile - m_tile * args.num_n_tiles;
      int ih0[8], iw0[8];
      long long off[8];
      uint32_t rowmask = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const long long m = static_cast<long long>(m_tile) * kBM + rsub + 16 * i;
        ih0[i] = 0;
        iw0[i] = 0;
        off[i] = 0;
        if (m < args.M) {
          const long long nimg = m / PQ;
          const int rem = static_cast<int>(m - nimg * PQ);
          const int p = rem / args.Q, q = rem - (rem / args.Q) * args.Q;
          ih0[i] = p * args.sh - args.pt;
          iw0[i] = q * args.sw - args.pl;
          off[i] = ((nimg * Hh + ih0[i]) * static_cast<long long>(Ww) + iw0[i]) * Cc;
          rowmask |= 1u << i;
        }
      }
      // (r, s, c) of this thread's chunk in k-block 0
      int c = j * 8, r = 0, s = 0;
      while (c >= Cc) {
        c -= Cc;
        if (++s == Ss) { s = 0; ++r; }
      }

      for (int kb = 0; kb < num_kb; ++kb) {
        if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, tmo)) {
          ok = false;
          break;
        }
        if (t == 0) {
          const uint32_t fb = smem_u32(&bars->full_b[stage]);
          mbar_arrive_expect_tx(fb, C::kBBytes);
          load_b_tile<BN>(smem_u32(sB + stage * C::kBBytes), &tmap_b, kb, n_tile, args.b3d, fb);
          ++issued;
        }
        const uint32_t a_base = smem_u32(sA + stage * C::kABytes);
        const bool kvalid = r < Rr;
        const long long koff = (static_cast<long long>(r) * Ww + s) * Cc + c;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ih = ih0[i] + r, iw = iw0[i] + s;
          const bool v = ((rowmask >> i) & 1u) && kvalid && static_cast<unsigned>(ih) < static_cast<unsigned>(Hh) &&
                         static_cast<unsigned>(iw) < static_cast<unsigned>(Ww);
          const uint16_t *src = v ? act + off[i] + koff : act;
          const int row = rsub + 16 * i;
          cp_async_16(a_base + row * 128 + ((j ^ (row & 7)) << 4), src, v ? 16u : 0u);
        }
        cp_async_commit();
        ++pending;
        if (pending > C::kLag) {
          cp_async_wait<C::kLag>();
          fence_proxy_async_smem();
          if (!drop) mbar_arrive(smem_u32(&bars->full_a[arr_stage]));
          if (++arr_stage == kStages) arr_stage = 0;
          --pending;
        }
        // advance this thread's chunk by 64 k-values
        c += kBK;
        while (c >= Cc) {
          c -= Cc;
          if (++s == Ss) { s = 0; ++r; }
        }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    while (pending > 0) {
      if (ok && !drop) mbar_arrive(smem_u32(&bars->full_a[arr_stage]));
      if (++arr_stage == kStages) arr_stage = 0;
      --pending;
    }
    if (t == 0) {
      // let any B-tile copy still in flight land before the CTA exits (after
      // an abort); on the normal path every one of them has completed
      const uint32_t first = issued > static_cast<uint32_t>(kStages) ? issued - kStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_drain(smem_u32(&bars->full_b[i % kStages]), (i / kStages) & 1u, 100000000ull);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform state); lane 0 issues.
    uint32_t stage = 0, phase = 0, astage = 0, aphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
      for (int kb0 = 0; kb0 < num_kb && ok; kb0 += kb_chunk) {
        const int kb1 = min(kb0 + kb_chunk, num_kb);
        if (!mbar_wait_warp(smem_u32(&bars->acc_empty[astage]), aphase ^ 1, abort_flag, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + astage * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_warp(smem_u32(&bars->full_a[stage]), phase, abort_flag, tmo) ||
              !mbar_wait_warp(smem_u32(&bars->full_b[stage]), phase, abort_flag, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::kABytes));
          const uint64_t bdesc = sw128_mnmajor_desc(smem_u32(sB + stage * C::kBBytes));
          if (lane == 0) {
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              umma_f16(d, adesc + 2 * k, bdesc + kBStepK * k, kIdesc,
                       (kb > kb0 || k > 0) ? 1u : 0u);
            umma_commit(smem_u32(&bars->empty[stage]));
          }
          __syncwarp();
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        if (lane == 0) umma_commit(smem_u32(&bars->acc_full[astage]));
        __syncwarp();
        if (++astage == 2) { astage = 0; aphase ^= 1; }
      }
    }
    if (lane == 0) {
      // every MMA issued above has completed once this arrives
      umma_commit(smem_u32(&bars->mma_done));
      mbar_wait_drain(smem_u32(&bars->mma_done), 0, 1000000000ull);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int ew = warp - kMmaWarp - 1;   // epilogue warp 0..3
    // this warp's copy of the tile columns' bias / scale, and its staging
    // buffer for the coalesced output stores
    float *wpar = reinterpret_cast<float *>(smem + C::kParamOffset) + ew * 2 * BN;
    uint4 *ostage = reinterpret_cast<uint4 *>(smem + C::kOutOffset) + ew * C::kOutWarpBytes / 16;
    uint32_t astage = 0, aphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < args.num_tiles && ok; tile += gridDim.x) {
      const int m_tile = tile / args.num_n_tiles;
      const int n_tile = tile - m_tile * args.num_n_tiles;
      const long long m = static_cast<long long>(m_tile) * kBM + row;
      const bool mvalid = m < args.M;
      const long long mo = out_pixel(args, m);   // the output pixel row m writes
      const int n0 = n_tile * BN;
      long long st_mo[SliceGroups<IS_INT8>::kGroups];
      bool st_ok[SliceGroups<IS_INT8>::kGroups];
      coalesced_rows<IS_INT8>(mo, mvalid, st_mo, st_ok);
      __syncwarp();   // every lane is done with the previous tile's copy
      if (args.mode == kModeFused && args.bias) {  // no bias when only the sums are written
        for (int j = lane; j < BN; j += 32) {
          const bool in = n0 + j < args.K;
          wpar[j] = in ? __ldg(args.bias + n0 + j) : 0.0f;
          if (args.scale_k) wpar[BN + j] = in ? __ldg(args.scale_k + n0 + j) : 0.0f;
        }
      }
      __syncwarp();
      const float *wscale = args.scale_k ? wpar + BN : nullptr;
      // the side input this thread reads after the tile's last chunk: into
      // L2 now, so the final epilogue does not wait on DRAM
      if (args.use_side && mvalid && n0 < args.K)
        prefetch_l2(static_cast<const uint8_t *>(args.side) + (mo * args.K + n0) * (IS_INT8 ? 1 : 2),
                    min(BN, args.K - n0) * (IS_INT8 ? 1 : 2));
      for (int ch = 0; ch < n_chunks; ++ch) {
        // one outcome for the whole warp: the stores below are warp-wide
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars->acc_full[astage]), aphase, abort_flag, tmo))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_off + astage * BN;
        const bool last = ch == n_chunks - 1;
#pragma unroll 1
        for (int jj = 0; jj < BN / 32; ++jj) {
          uint32_t v[32];
          tmem_ld32(t_acc + jj * 32, v);
          tmem_wait_ld(v);
          float vals[32];
          if (IS_INT8 && C::kCanChunk && n_chunks > 1) {
            // fold this chunk's exact fp32 sums into the int32 running sums
            const uint32_t t_sum = tmem_base + lane_off + 2 * BN + jj * 32;
            uint32_t sacc[32];
            if (ch > 0) {
              tmem_ld32(t_sum, sacc);
              tmem_wait_ld(sacc);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) sacc[i] = 0;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i)
              sacc[i] = static_cast<uint32_t>(static_cast<int>(sacc[i]) +
                                              __float2int_rn(__uint_as_float(v[i])));
            if (!last) {
              tmem_st32(t_sum, sacc);
              continue;
            }
            if (args.mode == kModeAccumulators) {
              if (mvalid) store_i32_slice(args, mo, n0 + jj * 32, sacc);
              continue;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) vals[i] = __int2float_rn(static_cast<int>(sacc[i]));
          } else {
            // bf16: + 0.0f turns a -0 sum into +0; int8: a zero of either
            // sign gives code 0 (and the raw int32 0), so it is skipped
#pragma unroll
            for (int i = 0; i < 32; ++i)
              vals[i] = IS_INT8 ? __uint_as_float(v[i]) : __fadd_rn(__uint_as_float(v[i]), 0.0f);
          }
          if (args.mode == kModeFused)
            epilogue_slice_warp<IS_INT8>(args, mo, mvalid, n0 + jj * 32, vals, nullptr,
                                         wpar + jj * 32, wscale ? wscale + jj * 32 : nullptr,
                                         ostage, st_mo, st_ok);
          else if (mvalid)
            store_raw_slice<IS_INT8>(args, mo, n0 + jj * 32, vals);
        }
        if (!last) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[astage]));
        if (++astage == 2) { astage = 0; aphase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem_base, C::kTmemCols);
}


// ---------------------------------------------------------------- TMA path
// Used when C % 64 == 0 (a k-block is 64 channels of one filter tap).
// 384 threads in three warpgroups.  Warpgroup 0: lane 0 of warp 0 issues
// the A loads (im2col) and lane 0 of warp 2 the B loads (tiled) of each
// stage onto the stage's full barrier; warp 1 allocates TMEM and lane 0
// issues the MMAs, with lane 0 of warp 3 issuing those of the second
// sub-tile on 256-pixel tiles (WIDEN: warp 0 issues both loads, warps 2-3
// widen the staged A, warp 1 issues every MMA).  Warpgroups 1-2
// (warps 4-11) run the epilogue, two warps per TMEM lane quarter, each owning
// half of the BN columns.  int8 sums longer than one exact chunk are folded
// into int32 registers of those threads, so all 512 TMEM columns hold a
// double-buffered 128 x 256 accumulator.
//
// Registers: the register file is split over the SM's four sub-partitions,
// so 12 warps launch at 168 a thread (384 x 168 = 64512).  Warpgroup 0 then
// gives back down to 40 and the epilogue warpgroups take 232:
// 128 x 40 + 256 x 232 = 64512, the launch total; per sub-partition that is
// one warp of each warpgroup, 40 + 232 + 232 = 504 <= 512 per lane.  ptxas
// allocates each region to its setmaxnreg budget: the int8 epilogue holds
// 128 int32 sums, 32 side words and a 32-column slice at once.  Tiles whose
// epilogue threads hold 64 sums or fewer split 96 / 200 instead
// (128 x 96 + 256 x 200 = 63488).
constexpr int kTmaThreads = 384;
constexpr int kTmaEpiWarp0 = 4;
constexpr int kTmaEpiWarps = 8;
// Register split by tile (see TmaCfg below): an int8 epilogue thread keeps
// kHalfCols int32 running sums; only tiles with 128 of them need 232
// registers there, and the others leave the control warps 96 (ptxas spills
// the 128-channel int8 instance's loop state at 40).
template <int HALF_COLS>
struct TmaRegs {
  static constexpr int kCtl = HALF_COLS >= 128 ? 40 : 96;
  static constexpr int kEpi = HALF_COLS >= 128 ? 232 : 200;
  static_assert(128 * kCtl + 256 * kEpi <= kTmaThreads * 168,
                "register split exceeds the launch allocation");
};

// MS: M sub-tiles of 128 output pixels per tile.  MS = 2 gives a tile of
// 256 pixels x BN channels whose two halves share each B stage (one B copy
// and one A walk per k-block for twice the MMA work, the MMAs from two
// issuing threads), for tiles narrower than 256 channels, where the issuing
// threads' fixed per-k-block work, not the tensor cores, sets the pace.
// WIDEN: int8 activations are loaded as they are (64 bytes a pixel) into a
// staging ring and widened to fp16 inside the kernel (see the converter
// role below), instead of being read from a widened copy in global memory.
// KPS: k-blocks a stage (2 on unchunked, unsplit 128-pixel tiles of up to
// 128 channels): a producer thread fills at most one stage per ~550-650
// cycles whatever the stage holds, so a stage of two k-blocks halves the
// producers' cost per k-block; the MMA issuer takes the stage's MMAs after
// one wait.
// HALO (the halo gather): instead of the stage ring a region of
// kHaloRegion bytes holds two input windows, two int8 window stagings and
// the CTA's whole filter tile, at offsets the plan gives (ConvArgs).
// KDUAL: two accumulators per tile, each k-block's k16 steps split between
// two MMA issuers (see the kernel); they are summed in the epilogue.
template <int BN, int MS = 1, bool WIDEN = false, int KPS = 1, bool HALO = false,
          bool KDUAL = false>
struct TmaCfg {
  static constexpr int kABytes = kBM * kBK * 2;        // one sub-tile's A of one k-block
  static constexpr int kAStage = HALO ? 0 : KPS * MS * kABytes;
  static constexpr int kBBytes = HALO ? 0 : KPS * BN * kBK * 2;
  static constexpr int kStageBytes = kAStage + kBBytes;
  // staging of the int8 A tiles (WIDEN): 128 pixels x 64 bytes a sub-tile
  static constexpr int kStgBytes = WIDEN ? MS * kBM * kBK : 0;
  static constexpr int kStgStages = WIDEN ? (MS == 2 ? 3 : 4) : 0;
  static constexpr int kStages0 =
      HALO ? 2 : (200 * 1024 - kStgStages * kStgBytes) / kStageBytes;
  static constexpr int kStages = HALO ? 2 : kStages0 > 8 ? 8 : kStages0;
  static constexpr int kAccCols = MS * BN * (KDUAL ? 2 : 1);   // one accumulator buffer
  static constexpr int kTmemCols = 2 * kAccCols <= 128 ? 128 : 2 * kAccCols <= 256 ? 256 : 512;
  static constexpr int kStgOffset = HALO ? kHaloRegion : kStages * kStageBytes;
  static constexpr int kBarOffset = kStgOffset + kStgStages * kStgBytes;
  // columns per epilogue thread: MS = 1 splits a row's BN columns between
  // two warps; MS = 2 gives each warp half one sub-tile's whole rows
  static constexpr int kHalfCols = MS == 1 ? BN / 2 : BN;
  static constexpr int kSlices = kHalfCols / 32;
  // after the barriers: each epilogue warp's copy of its columns' bias and
  // per-channel scale, [warp][bias | scale][kHalfCols] floats
  static constexpr int kParamOffset = kBarOffset + 256;
  static constexpr int kParamBytes = kTmaEpiWarps * 2 * kHalfCols * 4;
  // then each epilogue warp's output staging: 32 rows x 64 bytes (a bf16
  // slice; an int8 slice uses half)
  static constexpr int kOutOffset = kParamOffset + kParamBytes;
  static constexpr int kOutWarpBytes = 32 * 64;
  static constexpr int kSmemBytes = 1024 + kOutOffset + kTmaEpiWarps * kOutWarpBytes;
  static_assert(kSmemBytes <= 232448, "dynamic shared memory per block");
  static_assert(BN == 64 || BN == 128 || BN == 256, "TMA path tile");
  static_assert(MS == 1 || (MS == 2 && BN <= 128), "two sub-tiles need BN <= 128");
  static_assert(2 * kAccCols <= 512, "tensor memory");
  static_assert(HALO || kStages >= 3, "pipeline too shallow");
  static_assert(!HALO || (BN == 64 && !WIDEN && KPS == 1), "halo gather: 64-channel tiles");
  static_assert(!KDUAL || (MS == 1 && BN <= 128 && !WIDEN && !HALO),
                "split k16 steps: 128-pixel tiles of up to 128 channels");
  static_assert(!WIDEN || kHalfCols <= 64, "in-kernel widening needs the 96-register control warps");
  static_assert(KPS == 1 || (KPS == 2 && MS == 1 && !WIDEN), "two k-blocks a stage: 128-pixel tiles");
};

// SPLITK: the split-K form (units of kb_per_split k-blocks, partial sums
// and the last unit's reduction); the other instance keeps one unit a tile.
// WIDEN (int8, unsplit, BN <= 128): tmap_a is an im2col map of the int8
// input itself; warps 2-3 widen each staged A tile into the fp16 stage.
// HALO: the halo gather (see the loader role below): tmap_a is the tiled
// map of the input itself, the filter tile stays resident, unsplit.
// KDUAL: warps 1 and 3 both issue the MMAs of every k-block of a
// 128-pixel tile, warp 1 its first two k16 steps into accumulator 0, warp 3
// the last two into accumulator 1 (BN columns further); the epilogue adds
// the two.  One thread issues a tcgen05.mma about every 110 cycles, so a
// 128 x 128 tile's 4 MMAs a k-block take ~440 cycles from one thread
// against 256 cycles of tensor time; two threads issue 2 each.
template <int BN, bool IS_INT8, int MS, bool SPLITK, bool WIDEN = false, int KPS = 1,
          bool HALO = false, bool KDUAL = false>
__global__ void __launch_bounds__(kTmaThreads, 1)
    conv_fprop_tma_kernel(const __grid_constant__ CUtensorMap tmap_a,
                          const __grid_constant__ CUtensorMap tmap_b, const ConvArgs args) {
  static_assert(!WIDEN || (IS_INT8 && !SPLITK), "widening: int8, unsplit");
  static_assert(KPS == 1 || !SPLITK, "two k-blocks a stage: unsplit");
  static_assert(!HALO || !SPLITK, "halo gather: unsplit");
  static_assert(!KDUAL || !SPLITK, "split k16 steps: unsplit");
  using C = TmaCfg<BN, MS, WIDEN, KPS, HALO, KDUAL>;
  constexpr int kStages = C::kStages;
  constexpr uint32_t kIdesc = idesc_f16(kBM, BN, !IS_INT8, /*b_mn=*/true);
  constexpr int kTileM = kBM * MS;
  // Two MMA issuers (warps 1 and 3) for 256-pixel tiles: one thread issues a
  // tcgen05.mma no faster than about one per 105-120 cycles, while the
  // tensor core finishes a 128 x N x 16 MMA in about max(N / 2, 32 + N / 4)
  // cycles, so a single issuer leaves the tensor core idle on N <= 128.
  // Each issuer owns one 128-pixel sub-tile (its accumulator columns) and
  // commits to the stage and accumulator barriers, which then take two
  // arrivals.  (Splitting a 128-pixel tile's channels between two issuers,
  // N = BN / 2 each, measured slower on every 128 x 128 workload.)
  constexpr bool kDualMma = (!WIDEN && MS == 2) || KDUAL;
  constexpr int kMmaArrivals = kDualMma ? 2 : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;   // per stage: MS sub-tiles of A, 16 KB each (HALO: two windows)
  // HALO: the two int8 window stagings, then the resident filter tile
  uint8_t *sStgH = smem + (HALO ? 2 * args.halo_slot : 0);
  uint8_t *sB = HALO ? sStgH + 2 * args.halo_stg : smem + kStages * C::kAStage;
  uint8_t *sStg = smem + C::kStgOffset;   // WIDEN: the int8 A staging ring
  Smem *bars = reinterpret_cast<Smem *>(smem + C::kBarOffset);
  // WIDEN: the staging ring's barriers (the TMA kernel has no other use for
  // full_a): full_a[i] = staged tile i landed, full_a[4 + i] = slot i read
  uint64_t *stg_full = bars->full_a;
  uint64_t *stg_empty = bars->full_a + 4;
  volatile int *abort_flag = &bars->abort_flag;

  // taken from lane 0 so that the compiler sees a warp-uniform value and the
  // role branches below are uniform
  const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = args.timeout_ns;

  if (threadIdx.x == 0) {
    if constexpr (HALO) {
      // window buffer s: full_b[s] = ready for the MMA (bf16: its copy
      // landed; int8: both loader warps arrived, having widened their halves
      // or, for the first window, seen the epilogue warps widen it), empty[s] =
      // the MMAs that read it are done; int8 staging s: full_a[s] = a
      // window's copy landed, full_a[2 + s] = both widening warps have read
      // it; full_b[7] = the resident filter tile is in place (bf16: one
      // copy; int8: the 8 epilogue warps widened it)
      for (int s = 0; s < 2; ++s) {
        mbar_init(smem_u32(&bars->full_b[s]), IS_INT8 ? 2 : 1);
        mbar_init(smem_u32(&bars->empty[s]), kMmaArrivals);
        mbar_init(smem_u32(&bars->full_a[s]), 1);
        mbar_init(smem_u32(&bars->full_a[2 + s]), 2);
      }
      // int8: the epilogue warps widened the CTA's first window
      mbar_init(smem_u32(&bars->full_a[4]), kTmaEpiWarps);
      mbar_init(smem_u32(&bars->full_b[7]), IS_INT8 ? kTmaEpiWarps : 1);
    } else {
      for (int s = 0; s < kStages; ++s) {
        // the stage is full once both producers' copies have landed (A from
        // warp 0, B from warp 2); WIDEN: once the producer's B copy has
        // landed and both converter warps have written the A tile
        mbar_init(smem_u32(&bars->full_b[s]), WIDEN ? 3 : 2);
        mbar_init(smem_u32(&bars->empty[s]), kMmaArrivals);
      }
    }
    for (int i = 0; i < C::kStgStages; ++i) {
      mbar_init(smem_u32(&stg_full[i]), 1);
      mbar_init(smem_u32(&stg_empty[i]), 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&bars->acc_full[s]), kMmaArrivals);
      mbar_init(smem_u32(&bars->acc_empty[s]), kTmaEpiWarps);
    }
    mbar_init(smem_u32(&bars->mma_done), kMmaArrivals);
    bars->abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = __shfl_sync(0xffffffffu, bars->tmem_base, 0);

  const int num_kb = args.num_kb;
  const int splits = SPLITK ? args.splits : 1;
  const int kb_per_split = SPLITK ? args.kb_per_split : num_kb;
  const int kb_chunk = args.kb_chunk;

  if (warp < kTmaEpiWarp0) {
   setmaxnreg_dec<TmaRegs<C::kHalfCols>::kCtl>();
   if constexpr (HALO) {
    // ------------------------------------------------------------ halo gather
    // A tile is halo_tr whole output rows p0 .. of one image.  Its GEMM row
    // i = pr * Qh + q' (Qh = Q + S - 1) is output pixel (p0 + pr, q') when
    // q' < Q (other rows are computed and dropped), and its tap (r, s) reads
    // input pixel (p0 + pr + r - pt, q' + s - pl).  With the window of input
    // rows p0 - pt .. p0 - pt + halo_rows - 1 and columns -pl .. Qh - 1 - pl
    // stored pixel after pixel, that is window pixel i + r * Qh + s: every
    // tap's A operand is the window itself, shifted by r * Qh + s rows of
    // 128 bytes.  One tiled TMA copy a tile brings the window (zero outside
    // the image) in place of R * S im2col copies, and the CTA's filter tile
    // (all k-blocks of its output-channel tile: the grid is a multiple of
    // the channel tiles) is loaded once.
    const int Qh = args.halo_q;
    const int tiles_img = args.tiles_per_img;
    // one k-block a filter tap: 64 channels (C == 32: the upper 32 are the
    // window's zero fill and the filter tile's zero rows, and only the
    // first two k16 steps are issued)
    const int taps = args.R * args.S;
    const int ksteps = args.C / 16;
    auto window_origin = [&](long long unit, int &n_img, int &p0) {
      const int m_tile = static_cast<int>(unit / args.num_n_tiles);
      n_img = m_tile / tiles_img;
      p0 = (m_tile - n_img * tiles_img) * args.halo_tr;
    };
    const int win_px = args.halo_rows * Qh;   // window pixels
    if (warp == 0 || warp == 2) {
      // bf16: warp 0 copies the windows of the CTA's even tiles straight
      // into buffer 0, warp 2 those of its odd tiles into buffer 1, after
      // warp 2 has copied the filter tile.  int8: warp 0 copies window j
      // into staging j % 2 (window j + 1's copy is issued before window j is
      // widened, so it lands meanwhile), and both warps widen half of each
      // window's pixels into the tile's buffer.
      const int wi = warp >> 1;
      const bool drop = (args.debug & 1) != 0;
      if (!IS_INT8 && warp == 2) {
        if (lane == 0) {
          const uint32_t bb = smem_u32(&bars->full_b[7]);
          mbar_arrive_expect_tx(bb, static_cast<uint32_t>(taps) * BN * kBK * 2);
          const int n_tile = static_cast<int>(blockIdx.x) % args.num_n_tiles;
          for (int kb = 0; kb < taps; ++kb)
            load_b_tile<BN>(smem_u32(sB + kb * BN * kBK * 2), &tmap_b, kb, n_tile, args.b3d, bb);
        }
        __syncwarp();
      }
      const uint32_t win_bytes = static_cast<uint32_t>(win_px) * kBK * (IS_INT8 ? 1 : 2);
      // copies into window buffer / staging 0 and 1 (scalars: a runtime
      // index into a register array would put it in local memory)
      uint32_t issued0 = 0, issued1 = 0;
      if constexpr (IS_INT8) {
        bool ok = true;
        // warp 0: window jj's copy into staging jj % 2, once both warps have
        // read window jj - 2 from it
        auto issue = [&](long long jj) -> bool {
          const long long u = blockIdx.x + jj * gridDim.x;
          if (u >= args.num_tiles) return true;
          const int sb = static_cast<int>(jj & 1);
          const uint32_t sp = static_cast<uint32_t>(jj >> 1) & 1u;
          if (!mbar_wait_warp(smem_u32(&bars->full_a[2 + sb]), sp ^ 1, abort_flag, tmo))
            return false;
          if (!drop) {
            int n_img, p0;
            window_origin(u, n_img, p0);
            if (lane == 0) {
              const uint32_t sf = smem_u32(&bars->full_a[sb]);
              mbar_arrive_expect_tx(sf, win_bytes);
              tma_load_4d(smem_u32(sStgH + sb * args.halo_stg), &tmap_a, 0, -args.pl,
                          p0 - args.pt, n_img, sf);
            }
            __syncwarp();
            if (sb) ++issued1; else ++issued0;
          }
          return true;
        };
        if (warp == 0) ok = issue(0);
        for (long long j = 0; ok; ++j) {
          const long long unit = blockIdx.x + j * gridDim.x;
          if (unit >= args.num_tiles) break;
          if (warp == 0 && !issue(j + 1)) break;
          const int slot = static_cast<int>(j & 1);   // also the staging buffer
          const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
          if (!mbar_wait_warp(smem_u32(&bars->full_a[slot]), par, abort_flag, tmo) ||
              !mbar_wait_warp(smem_u32(&bars->empty[slot]), par ^ 1, abort_flag, tmo))
            break;
          if (j == 0) {
            // the epilogue warps widen the first window (see there)
            if (!mbar_wait_warp(smem_u32(&bars->full_a[4]), 0, abort_flag, tmo)) break;
          } else {
            const int half_px = (win_px + 1) / 2;
            widen_rows(sStgH + slot * args.halo_stg, sA + slot * args.halo_slot,
                       wi ? half_px : 0, wi ? win_px : half_px);
            fence_proxy_async_smem();   // the window is read by the tensor core
            __syncwarp();
          }
          if (lane == 0) {
            mbar_arrive(smem_u32(&bars->full_b[slot]));
            mbar_arrive(smem_u32(&bars->full_a[2 + slot]));
          }
        }
      } else {
        for (long long j = wi;; j += 2) {
          const long long unit = blockIdx.x + j * gridDim.x;
          if (unit >= args.num_tiles) break;
          const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
          if (!mbar_wait_warp(smem_u32(&bars->empty[wi]), par ^ 1, abort_flag, tmo)) break;
          if (!drop) {
            int n_img, p0;
            window_origin(unit, n_img, p0);
            if (lane == 0) {
              const uint32_t fb = smem_u32(&bars->full_b[wi]);
              mbar_arrive_expect_tx(fb, win_bytes);
              tma_load_4d(smem_u32(sA + wi * args.halo_slot), &tmap_a, 0, -args.pl,
                          p0 - args.pt, n_img, fb);
            }
            __syncwarp();
            if (wi) ++issued1; else ++issued0;
          }
        }
      }
      if (lane == 0) {
        // copies still in flight after an abort land before the CTA exits
        // (the last one into each buffer: a buffer's copies wait for each
        // other)
        if (issued0 > 0)
          mbar_wait_drain(smem_u32(IS_INT8 ? &bars->full_a[0] : &bars->full_b[0]),
                          (issued0 - 1) & 1u, 100000000ull);
        if (issued1 > 0)
          mbar_wait_drain(smem_u32(IS_INT8 ? &bars->full_a[1] : &bars->full_b[1]),
                          (issued1 - 1) & 1u, 100000000ull);
        if (!IS_INT8 && warp == 2) mbar_wait_drain(smem_u32(&bars->full_b[7]), 0, 100000000ull);
      }
      __syncwarp();
    } else if (warp == 1 || (kDualMma && warp == 3)) {
      // MMA issuer of sub-tile `part` of every tile (two issuers on
      // 256-pixel tiles): R * S k-blocks, each the window at its tap's shift
      // times that tap's resident filter block
      const int part = warp == 3 ? 1 : 0;
      bool ok = mbar_wait_warp(smem_u32(&bars->full_b[7]), 0, abort_flag, tmo);
      uint32_t astage = 0, aphase = 0;
      const uint32_t bbase = smem_u32(sB);
      for (long long j = 0; ok; ++j) {
        const long long unit = blockIdx.x + j * gridDim.x;
        if (unit >= args.num_tiles) break;
        const int slot = static_cast<int>(j & 1);
        const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
        if (!mbar_wait_warp(smem_u32(&bars->acc_empty[astage]), aphase ^ 1, abort_flag, tmo) ||
            !mbar_wait_warp(smem_u32(&bars->full_b[slot]), par, abort_flag, tmo))
          break;
        tc_fence_after();
        const uint32_t d = tmem_base + astage * C::kAccCols + part * BN;
        const uint32_t wbase = smem_u32(sA + slot * args.halo_slot);
        if (lane == 0) {
          int r = 0, s = 0;
          for (int kb = 0; kb < taps; ++kb) {
            const uint32_t row = static_cast<uint32_t>(part * kBM + r * Qh + s);
            const uint64_t adesc = sw128_kmajor_desc_at_row(wbase, row);
            const uint64_t bdesc = sw128_mnmajor_desc(bbase + kb * BN * kBK * 2);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              if (k < ksteps)
                umma_f16(d, adesc + 2 * k, bdesc + kBStepK * k, kIdesc,
                         (kb > 0 || k > 0) ? 1u : 0u);
            if (++s == args.S) { s = 0; ++r; }
          }
          umma_commit(smem_u32(&bars->empty[slot]));
          umma_commit(smem_u32(&bars->acc_full[astage]));
        }
        __syncwarp();
        if (++astage == 2) { astage = 0; aphase ^= 1; }
      }
      if (lane == 0) {
        // every MMA issued above has completed once this arrives
        umma_commit(smem_u32(&bars->mma_done));
        mbar_wait_drain(smem_u32(&bars->mma_done), 0, 1000000000ull);
      }
      __syncwarp();
    }
   } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop (warp-uniform state); lane 0 issues.
    const long long PQ = static_cast<long long>(args.P) * args.Q;
    const int cblocks = args.C / kBK;
    const bool drop = (args.debug & 1) != 0;
    griddep_wait();   // the widened input and filter copy of the prep launch
    uint32_t stage = 0, phase = 0, issued = 0;
    uint32_t sstage = 0, sphase = 0;   // WIDEN: the staging ring
    bool ok = true;
    const int num_units = args.num_tiles * splits;
    for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
      // unit: one split (a run of k-blocks) of one tile
      const int tile = unit / splits;
      const int ukb0 = (unit - tile * splits) * kb_per_split;
      const int ukb1 = min(num_kb, ukb0 + kb_per_split);
      const int m_tile = tile / args.num_n_tiles;
      const int n_tile = tile - m_tile * args.num_n_tiles;
      // filter-window origin of each sub-tile's first output pixel (a
      // sub-tile past the last pixel reads images beyond N: zero-filled)
      int w0[MS], h0[MS], n0[MS];
#pragma unroll
      for (int u = 0; u < MS; ++u) {
        const long long m0 = static_cast<long long>(m_tile) * kTileM + u * kBM;
        n0[u] = static_cast<int>(m0 / PQ);
        const int rem = static_cast<int>(m0 - static_cast<long long>(n0[u]) * PQ);
        const int p0 = rem / args.Q, q0 = rem - (rem / args.Q) * args.Q;
        w0[u] = q0 * args.sw - args.pl;
        h0[u] = p0 * args.sh - args.pt;
      }
      // filter tap and channel block of k-block kb (tap-major, channels fastest)
      int cb = ukb0 % cblocks, s = (ukb0 / cblocks) % args.S, r = ukb0 / cblocks / args.S;
      if constexpr (!WIDEN) {
        // A only: warp 2 copies each stage's B.  (Waiting for two free
        // stages and filling both in one pass measured slower: it gives up a
        // stage of lookahead.)
        for (int kb = ukb0; kb < ukb1; kb += KPS) {
          const int nk = KPS == 1 ? 1 : min(KPS, ukb1 - kb);   // the stage's k-blocks
          if (!mbar_wait_warp(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, tmo)) {
            ok = false;
            break;
          }
          if (!drop) {
            if (lane == 0) {
              // per k-block one copy of the tile's 128 * MS pixels: the
              // tensor map's walk length is the tile's, so a second
              // sub-tile continues the first one's walk
              const uint32_t fb = smem_u32(&bars->full_b[stage]);
              mbar_arrive_expect_tx(fb, nk * MS * C::kABytes);
              int cq = cb, sq = s, rq = r;
              for (int q = 0; q < nk; ++q) {
                tma_load_im2col_4d(smem_u32(sA + stage * C::kAStage + q * C::kABytes), &tmap_a,
                                   cq * kBK, w0[0], h0[0], n0[0], static_cast<uint16_t>(sq),
                                   static_cast<uint16_t>(rq), fb);
                if (++cq == cblocks) {
                  cq = 0;
                  if (++sq == args.S) { sq = 0; ++rq; }
                }
              }
            }
            __syncwarp();
            ++issued;
          }
          for (int q = 0; q < nk; ++q) {
            if (++cb == cblocks) {
              cb = 0;
              if (++s == args.S) { s = 0; ++r; }
            }
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
        }
      } else {
        for (int kb = ukb0; kb < ukb1; ++kb) {
          if (!mbar_wait_warp(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, tmo) ||
              !mbar_wait_warp(smem_u32(&stg_empty[sstage]), sphase ^ 1, abort_flag, tmo)) {
            ok = false;
            break;
          }
          if (!drop) {
            if (lane == 0) {
              // WIDEN: int8 A (64 bytes a pixel) into the staging slot, which
              // the converter warps widen into the stage, and the stage's B
              const uint32_t fb = smem_u32(&bars->full_b[stage]);
              const uint32_t sf = smem_u32(&stg_full[sstage]);
              mbar_arrive_expect_tx(sf, C::kStgBytes);
#pragma unroll
              for (int u = 0; u < MS; ++u)
                tma_load_im2col_4d(smem_u32(sStg + sstage * C::kStgBytes + u * kBM * kBK),
                                   &tmap_a, cb * kBK, w0[u], h0[u], n0[u],
                                   static_cast<uint16_t>(s), static_cast<uint16_t>(r), sf);
              mbar_arrive_expect_tx(fb, C::kBBytes);
              load_b_tile<BN>(smem_u32(sB + stage * C::kBBytes), &tmap_b, kb, n_tile, args.b3d,
                              fb);
            }
            __syncwarp();
            ++issued;
          }
          if (++cb == cblocks) {
            cb = 0;
            if (++s == args.S) { s = 0; ++r; }
          }
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          if (++sstage == C::kStgStages) { sstage = 0; sphase ^= 1; }
        }
      }
    }
    if (lane == 0) {
      // let any copy still in flight land before the CTA exits (after an
      // abort); on the normal path every one of them has completed
      const uint32_t first = issued > static_cast<uint32_t>(kStages) ? issued - kStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_drain(smem_u32(&bars->full_b[i % kStages]), (i / kStages) & 1u, 100000000ull);
      if constexpr (WIDEN) {
        const uint32_t sfirst =
            issued > static_cast<uint32_t>(C::kStgStages) ? issued - C::kStgStages : 0;
        for (uint32_t i = sfirst; i < issued; ++i)
          mbar_wait_drain(smem_u32(&stg_full[i % C::kStgStages]), (i / C::kStgStages) & 1u,
                          100000000ull);
      }
    }
    __syncwarp();
  } else if (!WIDEN && warp == 2) {
    // ------------------------------------------------------------ B producer
    // The filter tile of every k-block, into the same stages as warp 0's A
    // copies (each stage's full barrier takes both arrivals).  A producer's
    // stage rate is bound by the per-stage work of its issuing thread (the
    // barrier wait, the expect-tx arrival and each copy it issues), not by
    // the bytes, so two issuing warps fill stages faster than one.
    const bool drop = (args.debug & 1) != 0;
    griddep_wait();   // the filter copy of the prep launch
    uint32_t stage = 0, phase = 0, issued = 0;
    bool ok = true;
    const int num_units = args.num_tiles * splits;
    for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
      const int tile = unit / splits;
      const int ukb0 = (unit - tile * splits) * kb_per_split;
      const int ukb1 = min(num_kb, ukb0 + kb_per_split);
      const int n_tile = tile % args.num_n_tiles;
      for (int kb = ukb0; kb < ukb1; kb += KPS) {
        if (!mbar_wait_warp(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, tmo)) {
          ok = false;
          break;
        }
        if (!drop) {
          if (lane == 0) {
            // the stage's KPS k-blocks (a last stage of one k-block also
            // gets the next k-block's rows, or zeros past R*S*C: unused)
            const uint32_t fb = smem_u32(&bars->full_b[stage]);
            mbar_arrive_expect_tx(fb, C::kBBytes);
            load_b_tile<BN, KPS>(smem_u32(sB + stage * C::kBBytes), &tmap_b, kb, n_tile,
                                 args.b3d, fb);
          }
          __syncwarp();
          ++issued;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
    }
    if (lane == 0) {
      // let any copy still in flight land before the CTA exits
      const uint32_t first = issued > static_cast<uint32_t>(kStages) ? issued - kStages : 0;
      for (uint32_t i = first; i < issued; ++i)
        mbar_wait_drain(smem_u32(&bars->full_b[i % kStages]), (i / kStages) & 1u, 100000000ull);
    }
    __syncwarp();
  } else if (WIDEN && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------ converters
    // Widen each staged int8 A tile into the fp16 stage the MMA reads, in the
    // 128-byte-swizzled K-major layout a TMA copy would have written: staged
    // row r (a pixel, 64 bytes) becomes stage row r (128 bytes), its 16-byte
    // chunk j at position j ^ (r & 7).  The two warps follow the producer's
    // k-block sequence; each widens half of the tile's 16-byte pieces, then
    // fences its writes to the async proxy and signals the stage full and
    // the staging slot free.
    const int ct = (warp - 2) * 32 + lane;   // 0..63
    uint32_t stage = 0, phase = 0, sstage = 0, sphase = 0;
    bool ok = true;
    const int num_units = args.num_tiles * splits;
    for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
      const int ukb0 = (unit % splits) * kb_per_split;
      const int ukb1 = min(num_kb, ukb0 + kb_per_split);
      for (int kb = ukb0; kb < ukb1; ++kb) {
        if (!mbar_wait_warp(smem_u32(&stg_full[sstage]), sphase, abort_flag, tmo) ||
            !mbar_wait_warp(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, tmo)) {
          ok = false;
          break;
        }
        const uint8_t *src = sStg + sstage * C::kStgBytes;
        uint8_t *dst = sA + stage * C::kAStage;
#pragma unroll
        for (int i = 0; i < MS * 8; ++i) {
          const int q = ct + 64 * i;            // piece: sub-tile u, row r, 16 bytes p
          const int u = q >> 9, r = (q >> 2) & 127, pc = q & 3;
          const uint4 in = *reinterpret_cast<const uint4 *>(src + u * (kBM * kBK) + r * 64 +
                                                            pc * 16);
          uint4 lo, hi;
          i8x4_to_f16x4(in.x, lo.x, lo.y);
          i8x4_to_f16x4(in.y, lo.z, lo.w);
          i8x4_to_f16x4(in.z, hi.x, hi.y);
          i8x4_to_f16x4(in.w, hi.z, hi.w);
          uint8_t *row = dst + u * C::kABytes + r * 128;
          *reinterpret_cast<uint4 *>(row + (((2 * pc) ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4 *>(row + (((2 * pc + 1) ^ (r & 7)) << 4)) = hi;
        }
        fence_proxy_async_smem();   // the stage is read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&bars->full_b[stage]));
          mbar_arrive(smem_u32(&stg_empty[sstage]));
        }
        if (++stage == kStages) { stage = 0; phase ^= 1; }
        if (++sstage == C::kStgStages) { sstage = 0; sphase ^= 1; }
      }
    }
  } else if (warp == 1 || (kDualMma && warp == 3)) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (warp-uniform state); lane 0 issues.
    // Two k-blocks (stages) per iteration: one wait round trip and one pass
    // of loop control for each group of MMAs.  kDualMma: warps 1 and 3 both
    // run this loop, each issuing its part of every k-block's MMAs.
    const int part = warp == 3 ? 1 : 0;
    uint32_t stage = 0, phase = 0, astage = 0, aphase = 0;
    bool ok = true;
    const int num_units = args.num_tiles * splits;
    for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
      const int ukb0 = (unit % splits) * kb_per_split;
      const int ukb1 = min(num_kb, ukb0 + kb_per_split);
      for (int kb0 = ukb0; kb0 < ukb1 && ok; kb0 += kb_chunk) {
        const int kb1 = min(kb0 + kb_chunk, ukb1);
        if (!mbar_wait_warp(smem_u32(&bars->acc_empty[astage]), aphase ^ 1, abort_flag, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + astage * C::kAccCols;   // sub-tile u at d + u * BN
        if constexpr (KPS > 1) {
          // one stage (KPS k-blocks) a wait; A k-block q of the stage is
          // 16 KB further, B k-block q 8 KB further within each 64-channel
          // block (blocks 8 KB * KPS apart)
          for (int kb = kb0; kb < kb1; kb += KPS) {
            const int nk = min(KPS, kb1 - kb);
            if (!mbar_wait_warp(smem_u32(&bars->full_b[stage]), phase, abort_flag, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::kAStage));
            const uint64_t bdesc =
                sw128_mnmajor_desc(smem_u32(sB + stage * C::kBBytes), 8192 * KPS);
            if (lane == 0) {
#pragma unroll
              for (int q = 0; q < KPS; ++q) {
                if (q < nk) {
                  // KDUAL: this issuer's half of the k16 steps, its own accumulator
                  constexpr int k_n = KDUAL ? kBK / 32 : kBK / 16;
                  const int k_0 = KDUAL ? part * k_n : 0;
                  const uint32_t dd = KDUAL ? d + part * BN : d;
#pragma unroll
                  for (int kk = 0; kk < k_n; ++kk) {
                    const int k = k_0 + kk;
                    umma_f16(dd, adesc + q * (C::kABytes >> 4) + 2 * k,
                             bdesc + q * (8192 >> 4) + kBStepK * k, kIdesc,
                             (kb > kb0 || q > 0 || kk > 0) ? 1u : 0u);
                  }
                }
              }
              umma_commit(smem_u32(&bars->empty[stage]));
            }
            __syncwarp();
            if (++stage == kStages) { stage = 0; phase ^= 1; }
          }
        } else {
          for (int kb = kb0; kb < kb1; kb += 2) {
            const bool pair = kb + 1 < kb1;
            const uint32_t stage1 = stage + 1 == kStages ? 0 : stage + 1;
            const uint32_t phase1 = stage1 == 0 ? phase ^ 1 : phase;
            if (!mbar_wait2_warp(smem_u32(&bars->full_b[stage]), phase,
                                 smem_u32(&bars->full_b[stage1]), phase1, pair, abort_flag, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t adesc = sw128_kmajor_desc(smem_u32(sA + stage * C::kAStage));
            const uint64_t bdesc = sw128_mnmajor_desc(smem_u32(sB + stage * C::kBBytes));
            const uint64_t adesc1 = sw128_kmajor_desc(smem_u32(sA + stage1 * C::kAStage));
            const uint64_t bdesc1 = sw128_mnmajor_desc(smem_u32(sB + stage1 * C::kBBytes));
            // a sub-tile's A is 16 KB further: + (16384 >> 4) in the descriptor
            constexpr uint64_t kSubStep = static_cast<uint64_t>(C::kABytes >> 4);
            if (lane == 0) {
              if constexpr (KDUAL) {
                // this issuer's half of the k16 steps, its own accumulator
  #pragma unroll
                for (int kk = 0; kk < kBK / 32; ++kk) {
                  const int k = part * (kBK / 32) + kk;
                  umma_f16(d + part * BN, adesc + 2 * k, bdesc + kBStepK * k, kIdesc,
                           (kb > kb0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(&bars->empty[stage]));
                if (pair) {
  #pragma unroll
                  for (int kk = 0; kk < kBK / 32; ++kk) {
                    const int k = part * (kBK / 32) + kk;
                    umma_f16(d + part * BN, adesc1 + 2 * k, bdesc1 + kBStepK * k, kIdesc, 1u);
                  }
                  umma_commit(smem_u32(&bars->empty[stage1]));
                }
              } else if constexpr (kDualMma && MS == 2) {
                // this issuer's 128-pixel sub-tile
  #pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                  umma_f16(d + part * BN, adesc + part * kSubStep + 2 * k, bdesc + kBStepK * k,
                           kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
                umma_commit(smem_u32(&bars->empty[stage]));
                if (pair) {
  #pragma unroll
                  for (int k = 0; k < kBK / 16; ++k)
                    umma_f16(d + part * BN, adesc1 + part * kSubStep + 2 * k,
                             bdesc1 + kBStepK * k, kIdesc, 1u);
                  umma_commit(smem_u32(&bars->empty[stage1]));
                }
              } else {
  #pragma unroll
                for (int u = 0; u < MS; ++u)
  #pragma unroll
                  for (int k = 0; k < kBK / 16; ++k)
                    umma_f16(d + u * BN, adesc + u * kSubStep + 2 * k, bdesc + kBStepK * k,
                             kIdesc, (kb > kb0 || k > 0) ? 1u : 0u);
                umma_commit(smem_u32(&bars->empty[stage]));
                if (pair) {
  #pragma unroll
                  for (int u = 0; u < MS; ++u)
  #pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                      umma_f16(d + u * BN, adesc1 + u * kSubStep + 2 * k, bdesc1 + kBStepK * k,
                               kIdesc, 1u);
                  umma_commit(smem_u32(&bars->empty[stage1]));
                }
              }
            }
            __syncwarp();
            if (pair) {
              stage = stage1 + 1 == kStages ? 0 : stage1 + 1;
              phase = stage == 0 ? phase1 ^ 1 : phase1;
            } else {
              stage = stage1;
              phase = phase1;
            }
          }
        }
        if (!ok) break;
        if (lane == 0) umma_commit(smem_u32(&bars->acc_full[astage]));
        __syncwarp();
        if (++astage == 2) { astage = 0; aphase ^= 1; }
      }
    }
    if (lane == 0) {
      // every MMA issued above has completed once this arrives
      umma_commit(smem_u32(&bars->mma_done));
      mbar_wait_drain(smem_u32(&bars->mma_done), 0, 1000000000ull);
    }
    __syncwarp();
   }
  } else {
    setmaxnreg_inc<TmaRegs<C::kHalfCols>::kEpi>();
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;              // TMEM lanes 32*quarter .. +31
    const int half = (warp - kTmaEpiWarp0) >> 2;  // MS = 1: which half of the BN columns;
                                                  // MS = 2: which sub-tile
    const int row = (MS == 2 ? half * kBM : 0) + quarter * 32 + lane;   // in the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int cbase = MS == 2 ? 0 : half * C::kHalfCols;        // first column, in the tile
    const int tcol = (MS == 2 ? half * BN : 0) + cbase;          // its TMEM column offset
    int32_t sums[IS_INT8 ? C::kHalfCols : 1];  // int32 running sums across chunks
    // this warp's copy of the bias / scale of its tile columns: read as
    // shared-memory broadcasts by the epilogue instead of global loads that
    // queue behind the output stores
    float *wpar = reinterpret_cast<float *>(smem + C::kParamOffset) +
                  (warp - kTmaEpiWarp0) * 2 * C::kHalfCols;
    // this warp's staging buffer for the coalesced output stores
    uint4 *ostage = reinterpret_cast<uint4 *>(smem + C::kOutOffset) +
                    (warp - kTmaEpiWarp0) * C::kOutWarpBytes / 16;
    const int ew = warp - kTmaEpiWarp0;
    const int num_units = args.num_tiles * splits;
    if constexpr (HALO && IS_INT8) {
      // (at kernel start the epilogue warps have no accumulator to read yet)
      // the CTA's filter tile, widened from the caller's int8 HWIO filter
      // into the MN-major 128-byte-swizzled blocks the MMA reads (k-row c of
      // tap kb: 64 output channels, 16-byte chunk j at j ^ (c & 7)); output
      // channels past K and input channels past C (C == 32) read as zero.
      // All of a thread's loads are issued before its stores.
      const int t = (warp - kTmaEpiWarp0) * 32 + lane;   // 0 .. 255
      const int n0 = (static_cast<int>(blockIdx.x) % args.num_n_tiles) * BN;
      const int pieces = args.R * args.S * kBK * 4;        // 16 bytes of int8 each
      for (int i0 = 0; i0 < pieces; i0 += 256 * 4) {
        uint4 in[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int i = i0 + g * 256 + t;
          const int krow = i >> 2, col = n0 + (i & 3) * 16;
          const int tap = krow >> 6, c = krow & (kBK - 1);
          in[g] = (i < pieces && col < args.K && c < args.C)
                      ? ldg_nc_v4(args.w_i8 + (static_cast<size_t>(tap) * args.C + c) * args.K + col)
                      : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int i = i0 + g * 256 + t;
          if (i < pieces) {
            const int krow = i >> 2, pc = i & 3, c = krow & (kBK - 1);
            uint4 lo, hi;
            i8x4_to_f16x4(in[g].x, lo.x, lo.y);
            i8x4_to_f16x4(in[g].y, lo.z, lo.w);
            i8x4_to_f16x4(in[g].z, hi.x, hi.y);
            i8x4_to_f16x4(in[g].w, hi.z, hi.w);
            uint8_t *row = sB + (krow >> 6) * (BN * kBK * 2) + c * 128;
            *reinterpret_cast<uint4 *>(row + (((2 * pc) ^ (c & 7)) << 4)) = lo;
            *reinterpret_cast<uint4 *>(row + (((2 * pc + 1) ^ (c & 7)) << 4)) = hi;
          }
        }
      }
      fence_proxy_async_smem();   // the filter tile is read by the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->full_b[7]));
      // then the CTA's first window (eight warps instead of the loader
      // warps' two: the tensor core waits for it), once its copy has landed;
      // full_a[4] counts the warps done with it.  A wait that runs out skips
      // the widening: the loader warps' wait for full_a[4] runs out too.
      if (mbar_wait_warp(smem_u32(&bars->full_a[0]), 0, abort_flag, tmo)) {
        const int win_px = args.halo_rows * args.halo_q;
        const int per = (win_px + kTmaEpiWarps - 1) / kTmaEpiWarps;
        const int p0 = min(win_px, ew * per), p1 = min(win_px, p0 + per);
        widen_rows(sStgH, sA, p0, p1);
        fence_proxy_async_smem();   // the window is read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->full_a[4]));
      }
    }
    // split-K: the prep launch zeroes the completion counters.  The counter
    // atomics below already follow the producer's wait for that launch
    // (through the stage and accumulator barriers), but they wait for it
    // themselves too, which costs nothing by the time a unit is done.
    if (SPLITK) griddep_wait();
    uint32_t astage = 0, aphase = 0;
    bool ok = true;
    int wpar_c0 = -1;   // the columns whose bias / scale wpar holds
    for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
      const int tile = unit / splits;
      const int ukb0 = (unit - tile * splits) * kb_per_split;
      const int uchunks = (min(num_kb, ukb0 + kb_per_split) - ukb0 + kb_chunk - 1) / kb_chunk;
      // split-K: this unit's block of partial sums (this warp's rows and
      // columns; slice jj, 4-column group g, lane l at ((jj*8 + g)*32 + l)*4)
      uint32_t *const wpart =
          args.partial + (static_cast<size_t>(unit) * kTmaEpiWarps + ew) * 32 * C::kHalfCols;
      const int m_tile = tile / args.num_n_tiles;
      const int n_tile = tile - m_tile * args.num_n_tiles;
      const long long m = static_cast<long long>(m_tile) * kTileM + row;
      bool mvalid = m < args.M;
      long long mo;   // the output pixel row m writes
      if constexpr (HALO) {
        // pixel (pr, q') of the tile's output rows padded to halo_q columns
        const int n_img = m_tile / args.tiles_per_img;
        const int pr = row / args.halo_q, qv = row - pr * args.halo_q;
        const int pv = (m_tile - n_img * args.tiles_per_img) * args.halo_tr + pr;
        mvalid = pr < args.halo_tr && pv < args.P && qv < args.Q;
        mo = (static_cast<long long>(n_img) * args.P + pv) * args.Q + qv;
      } else {
        mo = out_pixel(args, m);
      }
      long long st_mo[SliceGroups<IS_INT8>::kGroups];
      bool st_ok[SliceGroups<IS_INT8>::kGroups];
      if (!HALO && !args.omap) {
        // output row = GEMM row: a warp's 32 rows are consecutive, so the
        // rows each lane stores follow without shuffles
        const long long m_lane0 = m - lane;
#pragma unroll
        for (int k = 0; k < SliceGroups<IS_INT8>::kGroups; ++k) {
          st_mo[k] = m_lane0 + (k * 32 + lane) / SliceGroups<IS_INT8>::kGroups;
          st_ok[k] = st_mo[k] < args.M;
        }
      } else {
        coalesced_rows<IS_INT8>(mo, mvalid, st_mo, st_ok);
      }
      const int c0 = n_tile * BN + cbase;
      // no bias when only the sums are written; a CTA whose units keep their
      // output-channel tile (the grid a multiple of the channel tiles) loads
      // it once
      if (args.mode == kModeFused && args.bias && c0 != wpar_c0) {
        __syncwarp();   // every lane is done with the previous tile's values
        for (int j = lane; j < C::kHalfCols; j += 32) {
          const bool in = c0 + j < args.K;
          wpar[j] = in ? __ldg(args.bias + c0 + j) : 0.0f;
          if (args.scale_k) wpar[C::kHalfCols + j] = in ? __ldg(args.scale_k + c0 + j) : 0.0f;
        }
        wpar_c0 = c0;
      }
      __syncwarp();   // every lane is done with the previous tile's copy
      const float *wscale = args.scale_k ? wpar + C::kHalfCols : nullptr;
      // the side input this thread reads after the tile's last chunk: into
      // L2 now, so the final epilogue does not wait on DRAM
      if (args.use_side && mvalid && c0 < args.K)
        prefetch_l2(static_cast<const uint8_t *>(args.side) + (mo * args.K + c0) * (IS_INT8 ? 1 : 2),
                    min(C::kHalfCols, args.K - c0) * (IS_INT8 ? 1 : 2));
      // the side words of the whole row segment, loaded before the wait for
      // the accumulator the outputs come from, so their latency overlaps it
      constexpr int kSideWords = C::kSlices * SliceGroups<IS_INT8>::kGroups;
      uint4 side_pre[kSideWords];
      const bool preload = args.use_side && mvalid && args.mode == kModeFused && splits == 1;
      // split-K: count this warp's partial in; the last unit of the tile
      // portion to arrive adds all partials in split order and stores
      auto finish_split = [&]() {
        __threadfence();   // this lane's partial words before the count
        __syncwarp();
        int* const counter = args.counters + tile * kTmaEpiWarps + ew;
        int old = 0;
        if (lane == 0) old = atomicAdd(counter, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old != splits - 1) return;   // a later unit finishes this portion
        if (lane == 0) atomicExch(counter, 0);   // zero again for the next run
        __threadfence();   // the other units' partial words after the count
        __syncwarp();
        const uint32_t *part0 =
            args.partial + (static_cast<size_t>(tile) * splits * kTmaEpiWarps + ew) * 32 *
                               C::kHalfCols;
        const size_t split_words = static_cast<size_t>(kTmaEpiWarps) * 32 * C::kHalfCols;
        auto add4 = [](uint4 &acc, const uint4 &q) {
          if (IS_INT8) {   // int32 sums: exact in any order
            acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
          } else {         // fp32 sums: added in split order
            acc.x = __float_as_uint(__fadd_rn(__uint_as_float(acc.x), __uint_as_float(q.x)));
            acc.y = __float_as_uint(__fadd_rn(__uint_as_float(acc.y), __uint_as_float(q.y)));
            acc.z = __float_as_uint(__fadd_rn(__uint_as_float(acc.z), __uint_as_float(q.z)));
            acc.w = __float_as_uint(__fadd_rn(__uint_as_float(acc.w), __uint_as_float(q.w)));
          }
        };
#pragma unroll 1
        for (int jj = 0; jj < C::kSlices; ++jj) {
          // a slice's 8 groups of two splits at a time in flight (16 loads
          // before the first add), added in split order
          const uint32_t *sl = part0 + static_cast<size_t>(jj * 8 * 32 + lane) * 4;
          uint4 acc[8];
#pragma unroll
          for (int g = 0; g < 8; ++g) acc[g] = ldcg_v4(sl + g * 128);
          int j = 1;
          for (; j + 1 < splits; j += 2) {
            uint4 q0[8], q1[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) q0[g] = ldcg_v4(sl + j * split_words + g * 128);
#pragma unroll
            for (int g = 0; g < 8; ++g) q1[g] = ldcg_v4(sl + (j + 1) * split_words + g * 128);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              add4(acc[g], q0[g]);
              add4(acc[g], q1[g]);
            }
          }
          if (j < splits) {
            uint4 q0[8];
#pragma unroll
            for (int g = 0; g < 8; ++g) q0[g] = ldcg_v4(sl + j * split_words + g * 128);
#pragma unroll
            for (int g = 0; g < 8; ++g) add4(acc[g], q0[g]);
          }
          uint32_t t[32];
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            t[4 * g + 0] = acc[g].x; t[4 * g + 1] = acc[g].y;
            t[4 * g + 2] = acc[g].z; t[4 * g + 3] = acc[g].w;
          }
          float vals[32];
#pragma unroll
          for (int i = 0; i < 32; ++i)
            vals[i] = IS_INT8 ? __int2float_rn(static_cast<int>(t[i]))
                              : __fadd_rn(__uint_as_float(t[i]), 0.0f);
          if (args.mode == kModeAccumulators) {
            if (mvalid) {
              if (IS_INT8) store_i32_slice(args, mo, c0 + jj * 32, t);
              else store_raw_slice<IS_INT8>(args, mo, c0 + jj * 32, vals);
            }
          } else {
            epilogue_slice_warp<IS_INT8>(args, mo, mvalid, c0 + jj * 32, vals, nullptr,
                                         wpar + jj * 32, wscale ? wscale + jj * 32 : nullptr,
                                         ostage, st_mo, st_ok);
          }
        }
      };
      for (int ch = 0; ch < uchunks; ++ch) {
        if (ch == uchunks - 1 && preload) {
#pragma unroll
          for (int jj = 0; jj < C::kSlices; ++jj)
            load_side_words<IS_INT8>(args, mo, c0 + jj * 32,
                                     side_pre + jj * SliceGroups<IS_INT8>::kGroups);
        }
        // one outcome for the whole warp: the stores below are warp-wide
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars->acc_full[astage]), aphase, abort_flag, tmo))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_acc = tmem_base + lane_off + astage * C::kAccCols + tcol;
        // 32 columns of this thread's row: KDUAL adds the second accumulator
        // (BN columns further) in fp32, exactly for int8 sums (integers whose
        // total stays below 2^24 within a chunk)
        auto acc_ld = [&](uint32_t taddr, uint32_t (&v)[32]) {
          tmem_ld32(taddr, v);
          if constexpr (KDUAL) {
            uint32_t v2[32];
            tmem_ld32(taddr + BN, v2);
            tmem_wait_ld(v);
            tmem_wait_ld(v2);
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = __float_as_uint(__fadd_rn(__uint_as_float(v[i]), __uint_as_float(v2[i])));
          } else {
            tmem_wait_ld(v);
          }
        };
        if (SPLITK && uchunks == 1) {
          // split-K, one chunk: the unit's sums (int32 for int8 plans, exact
          // here) from TMEM to its partial block, then the count
#pragma unroll
          for (int jj = 0; jj < C::kSlices; ++jj) {
            uint32_t v[32];
            tmem_ld32(t_acc + jj * 32, v);
            tmem_wait_ld(v);
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = IS_INT8 ? static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[4 * g + e])))
                                : v[4 * g + e];
              stg_v4(wpart + ((jj * 8 + g) * 32 + lane) * 4, make_uint4(w4[0], w4[1], w4[2], w4[3]));
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[astage]));
          finish_split();
        } else if (uchunks == 1) {
          // the whole sum is in TMEM: epilogue straight from it
          auto slice = [&](int jj, const uint4 *side_words) {
            uint32_t v[32];
            acc_ld(t_acc + jj * 32, v);
            float vals[32];
            // bf16: + 0.0f turns a -0 sum into +0; int8: a zero of either
            // sign gives code 0 (and the raw int32 0), so it is skipped
#pragma unroll
            for (int i = 0; i < 32; ++i)
              vals[i] = IS_INT8 ? __uint_as_float(v[i]) : __fadd_rn(__uint_as_float(v[i]), 0.0f);
            if (args.mode == kModeFused)
              epilogue_slice_warp<IS_INT8>(args, mo, mvalid, c0 + jj * 32, vals, side_words,
                                           wpar + jj * 32, wscale ? wscale + jj * 32 : nullptr,
                                           ostage, st_mo, st_ok);
            else if (mvalid)
              store_raw_slice<IS_INT8>(args, mo, c0 + jj * 32, vals);
          };
          // The branch must be the same for the whole warp (the slice code
          // is warp-collective), so it tests the plan, not this lane's row:
          // preload also depends on whether the lane's row exists.
          if (args.use_side && args.mode == kModeFused && splits == 1) {
            // side words preloaded per slice: static indexes
#pragma unroll
            for (int jj = 0; jj < C::kSlices; ++jj)
              slice(jj, preload ? side_pre + jj * SliceGroups<IS_INT8>::kGroups : nullptr);
          } else {
            // one copy of the slice code for all slices: the unrolled form
            // is kSlices times the instruction footprint of an epilogue
            // whose warps wait on instruction fetch between tiles
#pragma unroll 1
            for (int jj = 0; jj < C::kSlices; ++jj) slice(jj, nullptr);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[astage]));
        } else if constexpr (IS_INT8) {
          // fold this chunk's exact fp32 sums into the int32 registers, hand
          // the accumulator back, and finish the tile from the registers
#pragma unroll
          for (int jj = 0; jj < C::kSlices; ++jj) {
            uint32_t v[32];
            acc_ld(t_acc + jj * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int add = __float2int_rn(__uint_as_float(v[i]));
              sums[jj * 32 + i] = (ch == 0 ? 0 : sums[jj * 32 + i]) + add;
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->acc_empty[astage]));
          if (SPLITK && ch == uchunks - 1) {
            // split-K: the unit's int32 sums to its partial block, then the count
#pragma unroll
            for (int jj = 0; jj < C::kSlices; ++jj)
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                const int b = jj * 32 + 4 * g;
                stg_v4(wpart + ((jj * 8 + g) * 32 + lane) * 4,
                       make_uint4(static_cast<uint32_t>(sums[b]), static_cast<uint32_t>(sums[b + 1]),
                                  static_cast<uint32_t>(sums[b + 2]),
                                  static_cast<uint32_t>(sums[b + 3])));
              }
            finish_split();
          } else if (ch == uchunks - 1) {   // the whole warp: the fused stores are coalesced
#pragma unroll
            for (int jj = 0; jj < C::kSlices; ++jj) {
              if (args.mode == kModeAccumulators) {
                uint32_t u[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = static_cast<uint32_t>(sums[jj * 32 + i]);
                if (mvalid) store_i32_slice(args, mo, c0 + jj * 32, u);
              } else {
                float vals[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) vals[i] = __int2float_rn(sums[jj * 32 + i]);
                epilogue_slice_warp<IS_INT8>(args, mo, mvalid, c0 + jj * 32, vals,
                                             preload ? side_pre + jj * SliceGroups<IS_INT8>::kGroups
                                                     : nullptr,
                                             wpar + jj * 32, wscale ? wscale + jj * 32 : nullptr,
                                             ostage, st_mo, st_ok);
              }
            }
          }
        }
        if (++astage == 2) { astage = 0; aphase ^= 1; }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---------------------------------------------------------------- pre-pass
// One launch prepares the operands of a run: blocks [0, pack_blocks) write
// the 16-bit filter the B tiles are loaded from, [rows][K] in the HWIO
// order (int8 widened exactly to fp16; for a transposed plan the flipped
// taps, bf16 copied); the remaining blocks copy the input (int8 widened to
// fp16; subsampled or upsampled copies), 64 elements a thread per step.

constexpr int kPrepThreads = 256;

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv &d) {
  return (__umulhi(n, d.m) + n) >> d.l;
}

// Source of 8-element unit g of a subsampled or upsampled copy (-1: a zero
// unit): element 8g is channel c of copy pixel (n, a, b).  C is a multiple
// of 8 (16 for int8), so a unit never straddles two pixels and stays
// aligned; the copy holds fewer than 2^31 elements.
__device__ __forceinline__ long long copy_src_unit(long long g, const WidenMap &m) {
  const uint32_t u = static_cast<uint32_t>(g);
  const uint32_t pix = fast_div(u, m.units_per_pixel);
  const uint32_t cu = u - pix * m.units_per_pixel.d;
  const uint32_t n = fast_div(pix, m.pq);
  const uint32_t rem = pix - n * m.pq.d;
  const uint32_t a = fast_div(rem, m.q);
  const uint32_t b = rem - a * m.q.d;
  uint32_t h, w;
  if (m.mode == kCopySubsample) {
    h = a * static_cast<uint32_t>(m.sh);
    w = b * static_cast<uint32_t>(m.sw);
  } else {
    h = fast_div(a, m.div_sh);
    w = fast_div(b, m.div_sw);
    if (h * m.div_sh.d != a || w * m.div_sw.d != b) return -1;
  }
  return ((static_cast<long long>(n) * m.H + h) * m.W + w) * m.units_per_pixel.d + cu;
}

template <bool IS_INT8, bool MAPPED, int ROUNDS = 8>
__global__ void __launch_bounds__(kPrepThreads)
    prep_kernel(const void *__restrict__ w, uint16_t *__restrict__ wt, int rows, int K,
                int pack_blocks, const void *__restrict__ xv, __half *__restrict__ xh,
                long long n8, const WidenMap map, int *__restrict__ zero, int zero_n) {
  // the convolution launch behind this one may start its set-up now; it
  // waits for this grid before reading what it writes
  griddep_launch_dependents();
  if (blockIdx.x == 0)   // the split-K counters of the convolution
    for (int i = threadIdx.x; i < zero_n; i += kPrepThreads) zero[i] = 0;
  if (static_cast<int>(blockIdx.x) < pack_blocks) {
    // filter rows: packed row j of [rows][K] is row src(j) of the caller's
    // [R*S*C][K] filter (the same row for a forward plan; a flipped, for a
    // phase every stride-th, tap for a transposed plan), in 8-element
    // units (K is a multiple of 8; rows * K < 2^31)
    const uint32_t per_row = static_cast<uint32_t>(K) / 8;
    const uint32_t units = static_cast<uint32_t>(rows) * per_row;
    const uint32_t stride = static_cast<uint32_t>(pack_blocks) * kPrepThreads;
    // four units a pass, their loads in flight together before the stores
    constexpr int kPackUnroll = 4;
    for (uint32_t g0 = blockIdx.x * kPrepThreads + threadIdx.x; g0 < units;
         g0 += kPackUnroll * stride) {
      uint4 o[kPackUnroll];
      long long di[kPackUnroll];
#pragma unroll
      for (int k = 0; k < kPackUnroll; ++k) {
        const uint32_t g = g0 + k * stride;
        di[k] = -1;
        if (g >= units) continue;
        const uint32_t row = g / per_row, cu = g - row * per_row;
        uint32_t src = row;
        if (map.tap_nR > 0) {
          // (j, l, c) of the filter copy -> (r, s, c) of the caller's
          const int C = rows / (map.tap_nR * map.tap_nS);
          const int c = static_cast<int>(row) % C, jl = static_cast<int>(row) / C;
          const int j = jl / map.tap_nS, l = jl - j * map.tap_nS;
          const int r = map.tap_r0 + map.tap_rstep * (map.tap_nR - 1 - j);
          const int s2 = map.tap_s0 + map.tap_sstep * (map.tap_nS - 1 - l);
          src = static_cast<uint32_t>((r * map.tap_S + s2) * C + c);
        }
        const long long si = static_cast<long long>(src) * K + 8 * cu;
        di[k] = static_cast<long long>(row) * K + 8 * cu;
        if (IS_INT8) {
          const uint2 b8 =
              __ldg(reinterpret_cast<const uint2 *>(static_cast<const int8_t *>(w) + si));
          o[k] = make_uint4(b8.x, b8.y, 0u, 0u);   // widened below, after all loads
        } else {
          o[k] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(w) + si));
        }
      }
#pragma unroll
      for (int k = 0; k < kPackUnroll; ++k) {
        if (di[k] < 0) continue;
        uint4 v = o[k];
        if (IS_INT8) {
          i8x4_to_f16x4(o[k].x, v.x, v.y);
          i8x4_to_f16x4(o[k].y, v.z, v.w);
        }
        stg_v4(wt + di[k], v);
      }
    }
    return;
  }
  // Input copy, warp-contiguous: in one step a warp handles ROUNDS x 32
  // units of 8 elements; for each round lane l takes unit 32*round + l, so a
  // warp instruction loads 256 contiguous int8 bytes (or 512 bf16 bytes) of
  // a dense copy and stores 512 contiguous fp16 bytes, with all ROUNDS loads
  // in flight before the first store.  Subsampled and upsampled copies read
  // each unit from its own pixel (or write zeros).  Small copies take 2
  // rounds a step, so that their grid has enough warps to keep DRAM busy.
  constexpr int kStep = 32 * ROUNDS;
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x - pack_blocks) * (kPrepThreads / 32);
  for (long long base = (static_cast<long long>(blockIdx.x - pack_blocks) * (kPrepThreads / 32) +
                         (threadIdx.x >> 5)) * kStep;
       base < n8; base += warps * kStep) {
    if constexpr (IS_INT8) {
      const int8_t *x = static_cast<const int8_t *>(xv);
      uint2 in[ROUNDS];
#pragma unroll
      for (int u = 0; u < ROUNDS; ++u) {
        const long long g = base + u * 32 + lane;
        const long long src = MAPPED ? copy_src_unit(g, map) : g;
        // a zero byte widens to +0.0
        in[u] = (g < n8 && src >= 0) ? ldg_nc_v2(x + 8 * src) : make_uint2(0, 0);
      }
#pragma unroll
      for (int u = 0; u < ROUNDS; ++u) {
        const long long g = base + u * 32 + lane;
        if (g < n8) {
          uint4 o;
          i8x4_to_f16x4(in[u].x, o.x, o.y);
          i8x4_to_f16x4(in[u].y, o.z, o.w);
          stg_v4(xh + 8 * g, o);
        }
      }
    } else {
      const uint16_t *x = static_cast<const uint16_t *>(xv);
      uint4 in[ROUNDS];
#pragma unroll
      for (int u = 0; u < ROUNDS; ++u) {
        const long long g = base + u * 32 + lane;
        const long long src = MAPPED ? copy_src_unit(g, map) : g;
        in[u] = (g < n8 && src >= 0) ? ldg_nc_v4(x + 8 * src) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < ROUNDS; ++u) {
        const long long g = base + u * 32 + lane;
        if (g < n8) stg_v4(xh + 8 * g, in[u]);
      }
    }
  }
}

// int8 -> fp16 for the tail of an input whose size is not a multiple of 64
// (16 elements a thread; sizes are multiples of 16).
__global__ void widen_tail_kernel(const int8_t *__restrict__ x, __half *__restrict__ xh,
                                  long long first16, long long n16) {
  const long long i = first16 + blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  if (i >= n16) return;
  const uint4 in = ldg_nc_v4(x + 16 * i);
  uint4 o0, o1;
  i8x4_to_f16x4(in.x, o0.x, o0.y);
  i8x4_to_f16x4(in.y, o0.z, o0.w);
  i8x4_to_f16x4(in.z, o1.x, o1.y);
  i8x4_to_f16x4(in.w, o1.z, o1.w);
  stg_v4(xh + 16 * i, o0);
  stg_v4(xh + 16 * i + 8, o1);
}

// ---------------------------------------------------------------- launchers
// Raise a kernel's dynamic shared-memory limit once per device (the
// attribute call costs host time on every launch otherwise, and is best kept
// out of CUDA-graph captures).  `done` holds one bit per device ordinal.
template <typename Kern>
static cudaError_t ensure_smem_limit(Kern kern, int smem, std::atomic<unsigned long long> &done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// A convolution launch that may overlap the tail of the launch before it in
// the stream (programmatic stream serialization; the kernels wait for that
// grid before reading its output).  Only when that launch is this run's own
// prep launch (`overlap`): the kernels read the bias and per-channel scale
// before that wait, which the caller's own earlier kernels may still write.
template <typename... ExpTypes, typename... ActTypes>
static cudaError_t launch_overlapping(void (*kern)(ExpTypes...), bool overlap, int grid,
                                     int threads, int smem, cudaStream_t stream,
                                     ActTypes &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<ActTypes>(args)...);
}

template <int BN, bool IS_INT8>
static cudaError_t launch_cpasync_t(const CUtensorMap &tmap_b, const ConvArgs &args, int grid,
                                    bool overlap, cudaStream_t stream) {
  auto kern = conv_fprop_cpasync_kernel<BN, IS_INT8>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = ensure_smem_limit(kern, Cfg<BN>::kSmemBytes, configured);
  if (e == cudaSuccess) {
    e = launch_overlapping(kern, overlap, grid, kThreads, Cfg<BN>::kSmemBytes, stream, tmap_b,
                           args);
  }
  if (e != cudaSuccess) note_attributes(kern, kThreads, Cfg<BN>::kSmemBytes);
  return e;
}

// Attributes of the kernel a failed launch used, for the error message.
thread_local char t_kernel_note[256];

template <typename Kern>
static void note_attributes(Kern kern, int threads, int smem) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, kern) == cudaSuccess)
    snprintf(t_kernel_note, sizeof t_kernel_note,
             "kernel: %d registers, %zu B local, max %d threads/block; launch: %d threads, %d B "
             "dynamic shared memory",
             fa.numRegs, fa.localSizeBytes, fa.maxThreadsPerBlock, threads, smem);
}

const char *last_launch_note() { return t_kernel_note; }

template <int BN, bool IS_INT8, int MS, bool SPLITK = false, bool WIDEN = false, int KPS = 1,
          bool HALO = false, bool KDUAL = false>
static cudaError_t launch_tma_t(const CUtensorMap &tmap_a, const CUtensorMap &tmap_b,
                                const ConvArgs &args, int grid, bool overlap,
                                cudaStream_t stream) {
  auto kern = conv_fprop_tma_kernel<BN, IS_INT8, MS, SPLITK, WIDEN, KPS, HALO, KDUAL>;
  using Cfg = TmaCfg<BN, MS, WIDEN, KPS, HALO, KDUAL>;
  static std::atomic<unsigned long long> configured{0};
  cudaError_t e = ensure_smem_limit(kern, Cfg::kSmemBytes, configured);
  if (e == cudaSuccess) {
    e = launch_overlapping(kern, overlap, grid, kTmaThreads, Cfg::kSmemBytes, stream, tmap_a,
                           tmap_b, args);
  }
  if (e != cudaSuccess) note_attributes(kern, kTmaThreads, Cfg::kSmemBytes);
  return e;
}

bool gather_supports(Gather gather, int block_n, bool chunked, int m_sub) {
  if (m_sub != 1 && m_sub != 2) return false;
  if (gather == Gather::kTmaHalo) return block_n == 64 && !chunked;
  if (gather == Gather::kTmaIm2col)
    return m_sub == 1 ? (block_n == 64 || block_n == 128 || block_n == 256)
                      : (block_n == 64 || block_n == 128);
  if (m_sub != 1) return false;
  if (block_n != 64 && block_n != 128 && block_n != 256) return false;
  return !chunked || 3 * block_n <= 512;
}

cudaError_t launch_conv(int block_n, int m_sub, bool is_int8, Gather gather,
                        const CUtensorMap &tmap_a, const CUtensorMap &tmap_b,
                        const ConvArgs &args, int grid, bool overlap, cudaStream_t stream,
                        bool widen) {
  const bool chunked = args.kb_chunk < args.num_kb;
  if (chunked && !is_int8) return cudaErrorInvalidValue;
  if (!gather_supports(gather, block_n, chunked, m_sub)) return cudaErrorInvalidValue;
  if (args.kb_chunk <= 0 || grid <= 0) return cudaErrorInvalidValue;
  if (args.kps != 1 && (args.kps != 2 || widen || args.splits > 1 || m_sub != 1 ||
                        gather != Gather::kTmaIm2col))
    return cudaErrorInvalidValue;
  if (gather == Gather::kTmaHalo) {
    // the window and filter tile fit their buffers, a tile's output rows fit
    // its GEMM rows, and every CTA keeps one output-channel tile
    if (widen || args.splits != 1 || args.kps != 1 ||
        (args.C != kBK && !(is_int8 && args.C == 32)) || args.sh != 1 || args.sw != 1 ||
        args.R * args.S * block_n * kBK * 2 > kHaloBMax ||
        args.halo_q != args.Q + args.S - 1 || args.halo_q > 256 || args.halo_tr <= 0 ||
        args.halo_tr * args.halo_q > kBM * m_sub || args.halo_rows != args.halo_tr + args.R - 1 ||
        args.halo_rows > 256 || args.halo_slot % 1024 != 0 || args.halo_stg % 512 != 0 ||
        args.halo_rows * args.halo_q * 128 > args.halo_slot ||
        (is_int8 && args.halo_rows * args.halo_q * 64 > args.halo_stg) ||
        2 * args.halo_slot + 2 * args.halo_stg + args.R * args.S * block_n * kBK * 2 > kHaloRegion ||
        args.tiles_per_img != (args.P + args.halo_tr - 1) / args.halo_tr ||
        grid % args.num_n_tiles != 0 ||
        args.num_tiles != args.N * args.tiles_per_img * args.num_n_tiles ||
        (is_int8 && args.w_i8 == nullptr))
      return cudaErrorInvalidValue;
    if (m_sub == 2)
      return is_int8 ? launch_tma_t<64, true, 2, false, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                     : launch_tma_t<64, false, 2, false, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream);
    return is_int8 ? launch_tma_t<64, true, 1, false, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                   : launch_tma_t<64, false, 1, false, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream);
  }
  if (widen) {
    // int8 activations widened in the kernel: TMA gather, unsplit, <= 128 channels
    if (!is_int8 || gather != Gather::kTmaIm2col || args.splits > 1 || block_n > 128 ||
        args.C % kBK != 0)
      return cudaErrorInvalidValue;
    if (m_sub == 2) {   // 256-pixel tiles of 64 channels only (64 sums an epilogue thread)
      if (block_n != 64) return cudaErrorInvalidValue;
      return launch_tma_t<64, true, 2, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
    }
    return block_n == 64
               ? launch_tma_t<64, true, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream)
               : launch_tma_t<128, true, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
  }
  if (gather == Gather::kTmaIm2col && m_sub == 2) {
    if (args.C % kBK != 0) return cudaErrorInvalidValue;
    if (block_n == 64)
      return is_int8 ? launch_tma_t<64, true, 2>(tmap_a, tmap_b, args, grid, overlap, stream)
                     : launch_tma_t<64, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream);
    return is_int8 ? launch_tma_t<128, true, 2>(tmap_a, tmap_b, args, grid, overlap, stream)
                   : launch_tma_t<128, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream);
  }
  if (gather == Gather::kTmaIm2col && args.splits > 1) {
    // split-K: 128-pixel tiles of 64, 128 or 256 channels
    if (args.C % kBK != 0 || m_sub != 1 || block_n < 64 || args.partial == nullptr ||
        args.counters == nullptr || args.kb_per_split <= 0 ||
        (args.splits - 1) * args.kb_per_split >= args.num_kb)
      return cudaErrorInvalidValue;
    switch (block_n) {
      case 64: return is_int8 ? launch_tma_t<64, true, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                              : launch_tma_t<64, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream);
      case 128: return is_int8 ? launch_tma_t<128, true, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                               : launch_tma_t<128, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream);
      default: return is_int8 ? launch_tma_t<256, true, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                              : launch_tma_t<256, false, 1, true>(tmap_a, tmap_b, args, grid, overlap, stream);
    }
  }
  if (gather == Gather::kTmaIm2col && args.kdual) {
    // two MMA issuers splitting each k-block: unsplit 128-pixel tiles of <= 128 channels
    if (args.C % kBK != 0 || m_sub != 1 || args.splits != 1 || block_n > 128 ||
        (args.kps != 1 && args.kps != 2))
      return cudaErrorInvalidValue;
    if (args.kps == 2) {
      if (chunked) return cudaErrorInvalidValue;
      if (block_n == 64)
        return is_int8 ? launch_tma_t<64, true, 1, false, false, 2, false, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                       : launch_tma_t<64, false, 1, false, false, 2, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
      return is_int8 ? launch_tma_t<128, true, 1, false, false, 2, false, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                     : launch_tma_t<128, false, 1, false, false, 2, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
    }
    if (block_n == 64)
      return is_int8 ? launch_tma_t<64, true, 1, false, false, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                     : launch_tma_t<64, false, 1, false, false, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
    return is_int8 ? launch_tma_t<128, true, 1, false, false, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream)
                   : launch_tma_t<128, false, 1, false, false, 1, false, true>(tmap_a, tmap_b, args, grid, overlap, stream);
  }
  if (gather == Gather::kTmaIm2col && args.kps == 2) {
    // two k-blocks a stage: unsplit, unchunked 128-pixel tiles of <= 128 channels
    if (args.C % kBK != 0 || m_sub != 1 || chunked || block_n > 128)
      return cudaErrorInvalidValue;
    if (block_n == 64)
      return is_int8 ? launch_tma_t<64, true, 1, false, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream)
                     : launch_tma_t<64, false, 1, false, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream);
    return is_int8 ? launch_tma_t<128, true, 1, false, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream)
                   : launch_tma_t<128, false, 1, false, false, 2>(tmap_a, tmap_b, args, grid, overlap, stream);
  }
  if (gather == Gather::kTmaIm2col) {
    if (args.C % kBK != 0) return cudaErrorInvalidValue;
    switch (block_n) {
      case 64: return is_int8 ? launch_tma_t<64, true, 1>(tmap_a, tmap_b, args, grid, overlap, stream)
                              : launch_tma_t<64, false, 1>(tmap_a, tmap_b, args, grid, overlap, stream);
      case 128: return is_int8 ? launch_tma_t<128, true, 1>(tmap_a, tmap_b, args, grid, overlap, stream)
                               : launch_tma_t<128, false, 1>(tmap_a, tmap_b, args, grid, overlap, stream);
      default: return is_int8 ? launch_tma_t<256, true, 1>(tmap_a, tmap_b, args, grid, overlap, stream)
                              : launch_tma_t<256, false, 1>(tmap_a, tmap_b, args, grid, overlap, stream);
    }
  }
  switch (block_n) {
    case 64: return is_int8 ? launch_cpasync_t<64, true>(tmap_b, args, grid, overlap, stream)
                            : launch_cpasync_t<64, false>(tmap_b, args, grid, overlap, stream);
    case 128: return is_int8 ? launch_cpasync_t<128, true>(tmap_b, args, grid, overlap, stream)
                             : launch_cpasync_t<128, false>(tmap_b, args, grid, overlap, stream);
    default: return is_int8 ? launch_cpasync_t<256, true>(tmap_b, args, grid, overlap, stream)
                            : launch_cpasync_t<256, false>(tmap_b, args, grid, overlap, stream);
  }
}

static FastDiv make_fast_div(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, static_cast<uint32_t>(m), l};
}

cudaError_t launch_prep(bool is_int8, const void *w, uint16_t *wt, int rows, int K,
                        const void *x, __half *xh, long long n, const WidenMap &map_in,
                        int *zero, int zero_n, int sm_count, cudaStream_t stream) {
  WidenMap map = map_in;
  if (map.mode != kCopyDense) {
    if (map.C % 8 != 0 || map.P <= 0 || map.Q <= 0 || map.sh <= 0 || map.sw <= 0 ||
        n >= (1ll << 31))
      return cudaErrorInvalidValue;
    map.units_per_pixel = make_fast_div(static_cast<uint32_t>(map.C / 8));
    map.pq = make_fast_div(static_cast<uint32_t>(map.P) * static_cast<uint32_t>(map.Q));
    map.q = make_fast_div(static_cast<uint32_t>(map.Q));
    map.div_sh = make_fast_div(static_cast<uint32_t>(map.sh));
    map.div_sw = make_fast_div(static_cast<uint32_t>(map.sw));
  } else if (!is_int8) {
    n = 0;   // bf16 plans read a dense input as it is
  }
  // filter rows: 4 8-element units a thread (one pass), at most 8 blocks an SM
  const long long pack_units = w ? static_cast<long long>(rows) * (K / 8) : 0;
  long long pack_blocks_ll = (pack_units + 4 * kPrepThreads - 1) / (4 * kPrepThreads);
  if (pack_blocks_ll > 8LL * sm_count) pack_blocks_ll = 8LL * sm_count;
  const int pack_blocks = static_cast<int>(pack_blocks_ll);
  // 8-element units the main loop widens: all of a subsampled copy; the
  // whole 64-element groups of a dense one (the tail kernel does the rest)
  const long long n8 = map.mode != kCopyDense ? n / 8 : (n / 64) * 8;
  // 8 rounds a warp step (256 units), or 2 for copies too small to give each
  // SM 2 blocks that way: a 3.2 MB subsampled copy ran at ~5 % of the DRAM
  // peak on 1.3 blocks an SM (64x28x28x256 1x1/2: 16.4 -> 14.3 us a graph
  // step with 2 rounds; 32x7x7x512 7x7 VALID 40.1 -> 36.8), while copies
  // already at 2.6-5 blocks an SM ran slower with 4x as many blocks (the
  // 32x56x56x64 and 64x28x28x256 1x1 layers 18.5 -> 19.6, 32.8 -> 34.0: more
  // prep blocks hold the SMs the dependent convolution launch starts on)
  const long long step8_blocks = (n8 + 8 * kPrepThreads - 1) / (8 * kPrepThreads);
  const bool small = step8_blocks < 2LL * sm_count;
  const int rounds = small ? 2 : 8;
  long long widen_blocks = (n8 + rounds * kPrepThreads - 1) / (rounds * kPrepThreads);
  // up to 16 blocks an SM: more resident warps keep more loads in flight
  // (a cap of 4 an SM held the dense copy at ~81 % of the copy bandwidth,
  // 16 at ~96 %)
  const long long cap = static_cast<long long>(sm_count) * 16;
  if (widen_blocks > cap) widen_blocks = cap;
  unsigned grid = static_cast<unsigned>(pack_blocks + widen_blocks);
  if (grid == 0 && zero_n > 0) grid = 1;
  if (grid == 0) return cudaSuccess;
  const bool mapped = map.mode != kCopyDense;
  auto go = [&](auto kern) {
    kern<<<grid, kPrepThreads, 0, stream>>>(w, wt, rows, K, pack_blocks, x, xh, n8, map, zero,
                                            zero_n);
  };
  if (is_int8 && mapped)
    small ? go(prep_kernel<true, true, 2>) : go(prep_kernel<true, true, 8>);
  else if (is_int8)
    small ? go(prep_kernel<true, false, 2>) : go(prep_kernel<true, false, 8>);
  else if (mapped)
    small ? go(prep_kernel<false, true, 2>) : go(prep_kernel<false, true, 8>);
  else
    small ? go(prep_kernel<false, false, 2>) : go(prep_kernel<false, false, 8>);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || !is_int8 || map.mode != kCopyDense) return e;
  const long long n16 = n / 16, first16 = (n / 64) * 4;
  if (n16 > first16) {
    const long long rest = n16 - first16;
    widen_tail_kernel<<<static_cast<unsigned>((rest + 255) / 256), 256, 0, stream>>>(
        static_cast<const int8_t *>(x), xh, first16,
                                                                                     n16);
    e = cudaGetLastError();
  }
  return e;
}

cudaError_t status_read_and_clear(cudaStream_t stream, unsigned int *out) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(unsigned int), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  if (*out != 0) {
    e = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(unsigned int), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

}  // namespace fconv
