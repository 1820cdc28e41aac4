/*
 * CPU oracle for the fused quantized Conv2D forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code with the CUDA library.
 *
 * What it computes, and where the definition comes from
 * (page titles as printed at the top of each page):
 *
 *  - "conv_ops_fused_int8.cc" (TensorFlow), CPU helper
 *    LaunchFusedConv2DOpCpuInt8Helper: the fused op is a 2-D
 *    cross-correlation of an NHWC int8 input with an HWIO int8 filter,
 *    followed by the BiasActivationOutputKernel epilogue:
 *      (1) y = conv_output * conv_input_scale           (fp32, one rounding;
 *          conv_input_scale is a scalar, or one value per output channel
 *          when its tensor holds more than one element)
 *      (2) y = fmaf(side_input, side_input_scale, y)    (only if the side
 *          input is present and side_input_scale != 0; one rounding)
 *      (3) y = y + bias[k]                               (fp32, one rounding)
 *      then round half to even, clip to [lower, 127] with lower = -128 for
 *      BiasAdd and 0 for BiasAdd+Relu, and cast to int8.
 *    The page's comment on cuDNN 8 numerics fixes this order (multiply,
 *    then the side-input fma, then the bias add) and says the CPU path uses
 *    no packet FMA, so steps (1) and (3) are separately rounded.
 *  - Same page, GPU helper, comment "Total padding on rows and cols":
 *    SAME padding total Pr = max(0, (P-1)*stride + R - H); Pr/2 goes before
 *    and Pr - Pr/2 after (the extra pixel at the bottom/right).
 *  - "conv_grad_filter_ops.cc" (TensorFlow), function Im2col: patches in
 *    (h, w, c) storage order, taps outside the image are zero, and the
 *    output size is (H + pad_t + pad_b - R) / stride + 1.
 *
 *  - MIOpen's fusion page ("use-fusion-api"), tables "Convolution-based
 *    ... fusion for inference": the activations a fused plan may end with
 *    include Leaky Relu, Clipped Relu and CLAMP besides Relu.  The pages
 *    name them without formulas; the readings used here are the usual ones:
 *    leaky: y < 0 ? alpha*y : y (one fp32 rounding); clipped: min(max(y, 0),
 *    alpha); clamp: min(max(y, alpha), beta).  Each is applied after step
 *    (3), before the int8 rounding and clip to [-128, 127].
 *
 * Readings where the pages leave a step open:
 *  - The conv sum is accumulated exactly in int32 (the page's "QInt8xQInt8
 *    -> QInt32" contraction), and converted to fp32 with round-to-nearest-
 *    even before step (1).  The page's CPU path accumulates in fp32; the two
 *    agree whenever every partial sum is below 2^24 in magnitude.
 *  - The side input is skipped when it is absent or its scale is 0.0f.
 *  - The bf16 variant has no epilogue on the pages; its reference here runs
 *    the same three steps in fp64 on the exact values of the bf16 inputs,
 *    applies ReLU, and does not round the result.
 *
 * Build: cc -O3 -fopenmp -ffp-contract=off -fno-fast-math -fPIC -shared.
 * -ffp-contract=off keeps steps (1) and (3) as separate roundings; step (2)
 * calls fmaf() explicitly.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_SAME 0
#define ORC_VALID 1

/* Output extent and padding split along one spatial axis.
 * "conv_ops_fused_int8.cc", GPU helper, total-padding comment (SAME) and
 * "conv_grad_filter_ops.cc", Im2col output size (VALID and SAME).
 * Returns 0 on success, -1 if the arguments give no output. */
int orc_out_geometry(int in, int filt, int stride, int padding, int *out,
                     int *pad_before, int *pad_after) {
  if (in <= 0 || filt <= 0 || stride <= 0) return -1;
  if (padding == ORC_VALID) {
    if (filt > in) return -1;
    *out = (in - filt) / stride + 1;
    *pad_before = 0;
    *pad_after = 0;
    return 0;
  }
  if (padding != ORC_SAME) return -1;
  /* SAME: the output keeps ceil(in / stride) positions. */
  int o = (in + stride - 1) / stride;
  int total = (o - 1) * stride + filt - in;
  if (total < 0) total = 0;
  *out = o;
  *pad_before = total / 2;
  *pad_after = total - total / 2;
  return 0;
}

/* Direct convolution, int8 x int8 -> exact int32 sums.
 * x: NHWC [N][H][W][C]; w: HWIO [R][S][C][K]; acc: [N][P][Q][K].
 * acc[n,p,q,k] = sum over (r,s,c) with the input tap inside the image of
 * x[n, p*sh + r - pt, q*sw + s - pl, c] * w[r, s, c, k]
 * (cross-correlation, no filter flip; taps in the padding contribute zero).
 * The k loop is innermost only so that it runs over contiguous memory. */
void orc_conv_i8_direct(const int8_t *x, const int8_t *w, int N, int H, int W,
                        int C, int K, int R, int S, int sh, int sw, int pt,
                        int pl, int P, int Q, int32_t *acc) {
  long long NP = (long long)N * P;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long np = 0; np < NP; ++np) {
    int n = (int)(np / P), p = (int)(np % P);
    for (int q = 0; q < Q; ++q) {
      int32_t *a = acc + (((long long)n * P + p) * Q + q) * K;
      for (int k = 0; k < K; ++k) a[k] = 0;
      for (int r = 0; r < R; ++r) {
        int ih = p * sh + r - pt;
        if (ih < 0 || ih >= H) continue;
        for (int s = 0; s < S; ++s) {
          int iw = q * sw + s - pl;
          if (iw < 0 || iw >= W) continue;
          const int8_t *xp = x + (((long long)n * H + ih) * W + iw) * C;
          const int8_t *wp = w + ((long long)(r * S + s) * C) * K;
          for (int c = 0; c < C; ++c) {
            int32_t xv = xp[c];
            const int8_t *wr = wp + (long long)c * K;
            for (int k = 0; k < K; ++k) a[k] += xv * (int32_t)wr[k];
          }
        }
      }
    }
  }
}

/* The same sum for a list of single output elements (flat NPQK indices),
 * for sampling outputs of problems too large to evaluate whole. */
void orc_conv_i8_points(const int8_t *x, const int8_t *w, int N, int H, int W,
                        int C, int K, int R, int S, int sh, int sw, int pt,
                        int pl, int P, int Q, const int64_t *idx,
                        long long npts, int32_t *acc) {
  (void)N;
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < npts; ++t) {
    long long e = idx[t];
    int k = (int)(e % K);
    long long pix = e / K;
    int q = (int)(pix % Q);
    int p = (int)((pix / Q) % P);
    int n = (int)(pix / ((long long)P * Q));
    int32_t sum = 0;
    for (int r = 0; r < R; ++r) {
      int ih = p * sh + r - pt;
      if (ih < 0 || ih >= H) continue;
      for (int s = 0; s < S; ++s) {
        int iw = q * sw + s - pl;
        if (iw < 0 || iw >= W) continue;
        const int8_t *xp = x + (((long long)n * H + ih) * W + iw) * C;
        const int8_t *wp = w + ((long long)(r * S + s) * C) * K + k;
        for (int c = 0; c < C; ++c) sum += (int32_t)xp[c] * (int32_t)wp[(long long)c * K];
      }
    }
    acc[t] = sum;
  }
}

/* How large the partial sums of the int8 convolution get, for deciding
 * whether the page's CPU path, which accumulates in fp32
 * ("conv_ops_fused_int8.cc", LaunchFusedConv2DOpCpuInt8Helper with
 * TempT = float), reaches the same sums as the int32 reading.  Every
 * product is an integer, so an fp32 sum is exact while every value it
 * passes through is an integer below 2^24 in magnitude.  Over all outputs:
 *   bounds[0] = max |acc|                       (the final sums)
 *   bounds[1] = max |prefix sum|, the products added one at a time in the
 *               patch order (r, s, c) of the filter's [R*S*C][K] matrix:
 *               below 2^24, a sequential fp32 sum in that order is exact;
 *               below 2^23, so is any sum that adds contiguous runs of that
 *               order (a run is a difference of two prefixes)
 *   bounds[2] = max sum of |x * w|: below 2^24, every order is exact.
 * Same indexing and tap rule as orc_conv_i8_direct. */
void orc_conv_i8_partial_sums(const int8_t *x, const int8_t *w, int N, int H,
                              int W, int C, int K, int R, int S, int sh,
                              int sw, int pt, int pl, int P, int Q,
                              int64_t *bounds) {
  /* int32 running values: callers keep R*S*C below 2^17, so a sum of
   * |x * w| (each at most 2^14) stays below 2^31 */
  long long NP = (long long)N * P;
  int64_t g_acc = 0, g_pre = 0, g_abs = 0;
#pragma omp parallel
  {
    int64_t l_acc = 0, l_pre = 0, l_abs = 0;
    int32_t *a = (int32_t *)calloc((size_t)K * 3, sizeof(int32_t));
    int32_t *m = a + K, *t = a + 2 * (long long)K;
#pragma omp for schedule(dynamic, 1)
    for (long long np = 0; np < NP; ++np) {
      int n = (int)(np / P), p = (int)(np % P);
      for (int q = 0; q < Q; ++q) {
        for (int k = 0; k < K; ++k) a[k] = m[k] = t[k] = 0;
        for (int r = 0; r < R; ++r) {
          int ih = p * sh + r - pt;
          if (ih < 0 || ih >= H) continue;
          for (int s = 0; s < S; ++s) {
            int iw = q * sw + s - pl;
            if (iw < 0 || iw >= W) continue;
            const int8_t *xp = x + (((long long)n * H + ih) * W + iw) * C;
            const int8_t *wp = w + ((long long)(r * S + s) * C) * K;
            for (int c = 0; c < C; ++c) {
              int32_t xv = xp[c];
              const int8_t *wr = wp + (long long)c * K;
              for (int k = 0; k < K; ++k) {
                int32_t prod = xv * (int32_t)wr[k];
                int32_t sum = a[k] + prod;
                int32_t mag = sum < 0 ? -sum : sum;
                a[k] = sum;
                m[k] = mag > m[k] ? mag : m[k];
                t[k] += prod < 0 ? -prod : prod;
              }
            }
          }
        }
        for (int k = 0; k < K; ++k) {
          int64_t fin = a[k] < 0 ? -(int64_t)a[k] : a[k];
          if (fin > l_acc) l_acc = fin;
          if (m[k] > l_pre) l_pre = m[k];
          if (t[k] > l_abs) l_abs = t[k];
        }
      }
    }
#pragma omp critical
    {
      if (l_acc > g_acc) g_acc = l_acc;
      if (l_pre > g_pre) g_pre = l_pre;
      if (l_abs > g_abs) g_abs = l_abs;
    }
    free(a);
  }
  bounds[0] = g_acc;
  bounds[1] = g_pre;
  bounds[2] = g_abs;
}

/* Exact value of a bf16 bit pattern (bf16 is the top half of an fp32). */
static double bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Direct convolution of bf16 inputs (given as bit patterns), summed in fp64.
 * Same indexing as orc_conv_i8_direct. */
void orc_conv_bf16_direct_f64(const uint16_t *x, const uint16_t *w, int N,
                              int H, int W, int C, int K, int R, int S, int sh,
                              int sw, int pt, int pl, int P, int Q,
                              double *acc) {
  long long NP = (long long)N * P;
#pragma omp parallel for schedule(dynamic, 1)
  for (long long np = 0; np < NP; ++np) {
    int n = (int)(np / P), p = (int)(np % P);
    for (int q = 0; q < Q; ++q) {
      double *a = acc + (((long long)n * P + p) * Q + q) * K;
      for (int k = 0; k < K; ++k) a[k] = 0.0;
      for (int r = 0; r < R; ++r) {
        int ih = p * sh + r - pt;
        if (ih < 0 || ih >= H) continue;
        for (int s = 0; s < S; ++s) {
          int iw = q * sw + s - pl;
          if (iw < 0 || iw >= W) continue;
          const uint16_t *xp = x + (((long long)n * H + ih) * W + iw) * C;
          const uint16_t *wp = w + ((long long)(r * S + s) * C) * K;
          for (int c = 0; c < C; ++c) {
            double xv = bf16_value(xp[c]);
            const uint16_t *wr = wp + (long long)c * K;
            for (int k = 0; k < K; ++k) a[k] += xv * bf16_value(wr[k]);
          }
        }
      }
    }
  }
}

/* Sampled single elements of the bf16 fp64 sum. */
void orc_conv_bf16_points_f64(const uint16_t *x, const uint16_t *w, int N,
                              int H, int W, int C, int K, int R, int S, int sh,
                              int sw, int pt, int pl, int P, int Q,
                              const int64_t *idx, long long npts, double *acc) {
  (void)N;
#pragma omp parallel for schedule(static)
  for (long long t = 0; t < npts; ++t) {
    long long e = idx[t];
    int k = (int)(e % K);
    long long pix = e / K;
    int q = (int)(pix % Q);
    int p = (int)((pix / Q) % P);
    int n = (int)(pix / ((long long)P * Q));
    double sum = 0.0;
    for (int r = 0; r < R; ++r) {
      int ih = p * sh + r - pt;
      if (ih < 0 || ih >= H) continue;
      for (int s = 0; s < S; ++s) {
        int iw = q * sw + s - pl;
        if (iw < 0 || iw >= W) continue;
        const uint16_t *xp = x + (((long long)n * H + ih) * W + iw) * C;
        const uint16_t *wp = w + ((long long)(r * S + s) * C) * K + k;
        for (int c = 0; c < C; ++c)
          sum += bf16_value(xp[c]) * bf16_value(wp[(long long)c * K]);
      }
    }
    acc[t] = sum;
  }
}

/* Im2col for one NHWC image ("conv_grad_filter_ops.cc", Im2col): for each
 * output position (h, w) in raster order, the R*S*C patch in (r, s, c)
 * order; taps outside the image are zero.  elt = bytes per element.
 * col must hold P*Q*R*S*C elements. */
void orc_im2col(const void *image, int elt, int H, int W, int C, int R, int S,
                int pad_t, int pad_l, int pad_b, int pad_r, int sh, int sw,
                void *col) {
  const unsigned char *in = (const unsigned char *)image;
  unsigned char *out = (unsigned char *)col;
  int P = (H + pad_t + pad_b - R) / sh + 1;
  int Q = (W + pad_l + pad_r - S) / sw + 1;
  size_t row = (size_t)C * elt;
  for (int p = 0; p < P; ++p) {
    int h0 = p * sh - pad_t;
    for (int q = 0; q < Q; ++q) {
      int w0 = q * sw - pad_l;
      for (int ih = h0; ih < h0 + R; ++ih) {
        for (int iw = w0; iw < w0 + S; ++iw) {
          if (ih >= 0 && ih < H && iw >= 0 && iw < W)
            memcpy(out, in + ((size_t)ih * W + iw) * row, row);
          else
            memset(out, 0, row);
          out += row;
        }
      }
    }
  }
}

/* Plain GEMM C[M][N] = A[M][Kd] * B[Kd][N], int8 operands, int32 sums. */
void orc_gemm_i8(const int8_t *A, const int8_t *B, int M, int Kd, int N,
                 int32_t *Cm) {
#pragma omp parallel for schedule(static)
  for (int i = 0; i < M; ++i) {
    int32_t *c = Cm + (long long)i * N;
    for (int j = 0; j < N; ++j) c[j] = 0;
    for (int t = 0; t < Kd; ++t) {
      int32_t a = A[(long long)i * Kd + t];
      const int8_t *b = B + (long long)t * N;
      for (int j = 0; j < N; ++j) c[j] += a * (int32_t)b[j];
    }
  }
}

/* Convolution by im2col + GEMM, one image at a time: the filter HWIO
 * [R][S][C][K] is read as a [R*S*C][K] matrix, which matches the (r, s, c)
 * patch order.  col_scratch must hold P*Q*R*S*C bytes. */
void orc_conv_i8_im2col(const int8_t *x, const int8_t *w, int N, int H, int W,
                        int C, int K, int R, int S, int sh, int sw, int pt,
                        int pb, int pl, int pr, int32_t *acc,
                        int8_t *col_scratch) {
  int P = (H + pt + pb - R) / sh + 1;
  int Q = (W + pl + pr - S) / sw + 1;
  for (int n = 0; n < N; ++n) {
    orc_im2col(x + (long long)n * H * W * C, 1, H, W, C, R, S, pt, pl, pb, pr,
               sh, sw, col_scratch);
    orc_gemm_i8(col_scratch, w, P * Q, R * S * C, K,
                acc + (long long)n * P * Q * K);
  }
}

/* Transposed convolution ("cudnn_deconvolution-inl.h", MXNet, Forward: the
 * backward-data pass of the cross-correlation with the op's pad and stride,
 * then the bias).  Written as the scatter that defines that adjoint:
 *   out[n, p*sh + r - pt, q*sw + s - pl, k] += x[n, p, q, c] * w[r, s, c, k]
 * for every input pixel (p < H, q < W), tap (r, s) and channel pair whose
 * target lies inside the Ho x Wo output; Ho = (H - 1)*sh + R - pt - pb
 * (MXNet's symmetric pad p with output adjustment a: pt = p, pb = p - a).
 * x: NHWC [N][H][W][C]; w: [R][S][C][K] (C input, K output channels);
 * out: [N][Ho][Wo][K], exact int32 sums.  One image per thread: no races. */
void orc_convT_i8_direct(const int8_t *x, const int8_t *w, int N, int H, int W,
                         int C, int K, int R, int S, int sh, int sw, int pt,
                         int pl, int Ho, int Wo, int32_t *out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < N; ++n) {
    int32_t *o = out + (long long)n * Ho * Wo * K;
    for (long long i = 0; i < (long long)Ho * Wo * K; ++i) o[i] = 0;
    for (int p = 0; p < H; ++p) {
      for (int q = 0; q < W; ++q) {
        const int8_t *xp = x + (((long long)n * H + p) * W + q) * C;
        for (int r = 0; r < R; ++r) {
          int oh = p * sh + r - pt;
          if (oh < 0 || oh >= Ho) continue;
          for (int s2 = 0; s2 < S; ++s2) {
            int ow = q * sw + s2 - pl;
            if (ow < 0 || ow >= Wo) continue;
            int32_t *op = o + ((long long)oh * Wo + ow) * K;
            const int8_t *wp = w + ((long long)(r * S + s2) * C) * K;
            for (int c = 0; c < C; ++c) {
              int32_t xv = xp[c];
              const int8_t *wr = wp + (long long)c * K;
              for (int k = 0; k < K; ++k) op[k] += xv * (int32_t)wr[k];
            }
          }
        }
      }
    }
  }
}

/* The same scatter on bf16 inputs (bit patterns), summed in fp64. */
void orc_convT_bf16_direct_f64(const uint16_t *x, const uint16_t *w, int N,
                               int H, int W, int C, int K, int R, int S,
                               int sh, int sw, int pt, int pl, int Ho, int Wo,
                               double *out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int n = 0; n < N; ++n) {
    double *o = out + (long long)n * Ho * Wo * K;
    for (long long i = 0; i < (long long)Ho * Wo * K; ++i) o[i] = 0.0;
    for (int p = 0; p < H; ++p) {
      for (int q = 0; q < W; ++q) {
        const uint16_t *xp = x + (((long long)n * H + p) * W + q) * C;
        for (int r = 0; r < R; ++r) {
          int oh = p * sh + r - pt;
          if (oh < 0 || oh >= Ho) continue;
          for (int s2 = 0; s2 < S; ++s2) {
            int ow = q * sw + s2 - pl;
            if (ow < 0 || ow >= Wo) continue;
            double *op = o + ((long long)oh * Wo + ow) * K;
            const uint16_t *wp = w + ((long long)(r * S + s2) * C) * K;
            for (int c = 0; c < C; ++c) {
              double xv = bf16_value(xp[c]);
              const uint16_t *wr = wp + (long long)c * K;
              for (int k = 0; k < K; ++k) op[k] += xv * bf16_value(wr[k]);
            }
          }
        }
      }
    }
  }
}

/* The epilogue of BiasActivationOutputKernel ("conv_ops_fused_int8.cc"),
 * applied to rows x K exact int32 sums.  side may be NULL.  conv_scale_k is
 * NULL for a scalar conv_input_scale, else its K per-channel values (the
 * kernel's step (1) offsets the scale pointer by the output channel when the
 * scale tensor holds more than one element). */
/* Activation codes: 0 none (BiasAdd), 1 Relu, 2 leaky Relu (alpha),
 * 3 clipped Relu (alpha), 4 clamp to [alpha, beta]. */
#define ORC_ACT_NONE 0
#define ORC_ACT_RELU 1
#define ORC_ACT_LEAKY 2
#define ORC_ACT_CLIPPED 3
#define ORC_ACT_CLAMP 4

static float act_f32(float v, int act, float alpha, float beta) {
  switch (act) {
    case ORC_ACT_LEAKY: return v < 0.0f ? v * alpha : v;
    case ORC_ACT_CLIPPED:
      if (v < 0.0f) v = 0.0f;
      return v > alpha ? alpha : v;
    case ORC_ACT_CLAMP:
      if (v < alpha) v = alpha;
      return v > beta ? beta : v;
    default: return v;   /* none; Relu is the clip's lower bound */
  }
}

void orc_epilogue_i8(const int32_t *acc, long long rows, int K,
                     const float *bias, const int8_t *side, float conv_scale,
                     const float *conv_scale_k, float side_scale, int act,
                     float alpha, float beta, int8_t *out) {
  const float lower = act == ORC_ACT_RELU ? 0.0f : -128.0f;
  const float upper = 127.0f;
  const int use_side = (side != NULL) && (side_scale != 0.0f);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < rows; ++i) {
    for (int k = 0; k < K; ++k) {
      long long e = i * K + k;
      float v = (float)acc[e];          /* int32 -> fp32, round to nearest even */
      /* (1) scale: per output channel when a [K] vector is given */
      v = v * (conv_scale_k ? conv_scale_k[k] : conv_scale);
      if (use_side)                     /* (2) side input, one fused rounding */
        v = fmaf((float)side[e], side_scale, v);
      v = v + bias[k];                  /* (3) bias */
      v = act_f32(v, act, alpha, beta); /* activation other than Relu */
      float r = nearbyintf(v);          /* round half to even (default mode) */
      if (r < lower) r = lower;         /* clip to [lower, 127] */
      if (r > upper) r = upper;
      out[e] = (int8_t)r;
    }
  }
}

/* fp64 reference of the same three steps for the bf16 variant (no output
 * rounding).  side holds bf16 bit patterns and may be NULL. */
void orc_epilogue_f64(const double *acc, long long rows, int K,
                      const float *bias, const uint16_t *side,
                      double conv_scale, const float *conv_scale_k,
                      double side_scale, int act, double alpha, double beta,
                      double *out) {
  const int use_side = (side != NULL) && (side_scale != 0.0);
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < rows; ++i) {
    for (int k = 0; k < K; ++k) {
      long long e = i * K + k;
      double v = acc[e] * (conv_scale_k ? (double)conv_scale_k[k] : conv_scale);
      if (use_side) v = bf16_value(side[e]) * side_scale + v;
      v = v + (double)bias[k];
      switch (act) {
        case ORC_ACT_RELU: if (v < 0.0) v = 0.0; break;
        case ORC_ACT_LEAKY: if (v < 0.0) v = v * alpha; break;
        case ORC_ACT_CLIPPED: if (v < 0.0) v = 0.0; if (v > alpha) v = alpha; break;
        case ORC_ACT_CLAMP: if (v < alpha) v = alpha; if (v > beta) v = beta; break;
        default: break;
      }
      out[e] = v;
    }
  }
}

/* Number of OpenMP threads the oracle runs with. */
int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
