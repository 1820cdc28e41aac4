/*
 * fconv -- fused quantized Conv2D forward pass for GB300 (sm_103a).
 *
 * One operation, the vertically fused 2-D convolution forward pass of
 * TensorFlow's fused int8 kernel ("conv_ops_fused_int8.cc", the
 * LaunchFusedConv2DOp helpers and BiasActivationOutputKernel):
 *
 *   acc[n,p,q,k] = sum_{r,s,c} x[n, p*sh + r - pt, q*sw + s - pl, c] * w[r,s,c,k]
 *                  (cross-correlation; taps outside the image contribute 0)
 *   y = float(acc) * conv_scale                  (1) one fp32 rounding
 *   y = fmaf(float(side), side_scale, y)         (2) only if side != NULL and
 *                                                    side_scale != 0
 *   y = y + bias[k]                              (3) one fp32 rounding
 *   int8 out: clip(round_half_even(y), lower, 127), lower = -128 (BiasAdd)
 *             or 0 (BiasAdd + Relu)
 *   bf16 out: bf16_round_nearest_even(relu ? max(y, 0) : y)
 *
 * The order (1)(2)(3), each rounded once, is the one that page's epilogue
 * implements and its comment attributes to cuDNN 8 on sm75+.  int8 sums are
 * exact (int32 semantics); bf16 sums are fp32.
 *
 * Layouts (all row-major, densely packed):
 *   x    NHWC  [N][H][W][C]         int8 or bf16
 *   w    HWIO  [R][S][C][K]         same dtype as x
 *   bias [K]                        fp32
 *   side NHWC  [N][P][Q][K]         same dtype as the output (nullable)
 *   y    NHWC  [N][P][Q][K]         int8 or bf16
 * Output geometry follows the TensorFlow rule on the same page (the comment
 * on the total padding) and the Im2col output size of
 * "conv_grad_filter_ops.cc": SAME gives P = ceil(H / sh) with total padding
 * max(0, (P-1)*sh + R - H), of which the smaller half goes on top and the
 * odd pixel at the bottom (likewise left/right); VALID gives
 * P = (H - R) / sh + 1 and no padding.
 *
 * The plan lifecycle (create once, run many times with new pointers,
 * destroy) follows the fusion-plan workflow of MIOpen's "use-fusion-api"
 * page: plan creation validates and fixes the kernel configuration, runs
 * only bind buffers.
 *
 * Ownership and errors: the caller owns every buffer and the stream; a plan
 * owns only host memory (its settings and the TMA descriptors of its last
 * run, re-encoded when a tensor's address changes).  A plan is used by one
 * host thread at a time; different plans are independent.  Runs capture
 * into CUDA graphs (after one run outside the capture on that device).
 * Every call returns a status and never aborts.
 * Device pointers must be device-accessible memory of the current device.
 * Runs are asynchronous on the given stream; a kernel that gives up waiting
 * (a stalled pipeline) records FCONV_ERR_TIMEOUT in a per-device word that
 * fconv_plan_check() reads.
 */
#ifndef FCONV_H_
#define FCONV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct fconv_plan fconv_plan;
/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fconv_stream_t;

typedef enum {
  FCONV_OK = 0,
  FCONV_ERR_INVALID_VALUE = 1, /* bad dimension, NULL required pointer, ... */
  FCONV_ERR_NOT_SUPPORTED = 2, /* valid convolution this library does not run */
  FCONV_ERR_MISALIGNED = 3,    /* pointer or channel count breaks 16-byte rule */
  FCONV_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed */
  FCONV_ERR_TIMEOUT = 5,       /* a kernel gave up on a pipeline wait */
  FCONV_ERR_INTERNAL = 6,
  FCONV_ERR_WORKSPACE = 7      /* workspace missing or smaller than required */
} fconv_status;

typedef enum { FCONV_SAME = 0, FCONV_VALID = 1 } fconv_padding;
typedef enum { FCONV_INT8 = 0, FCONV_BF16 = 1 } fconv_dtype;
/* Activation after the bias add.  BiasAdd (NONE) and BiasAdd+Relu are the
 * two fusions the TensorFlow kernel accepts ("conv_ops_fused_int8.cc");
 * MIOpen's fusion tables ("use-fusion-api", convolution-based fusion for
 * inference) also list leaky Relu, clipped Relu and CLAMP, which the pages
 * name without formulas.  Read here as, on the fp32 value y after step (3):
 *   LEAKY_RELU:   y < 0 ? alpha * y : y   (one fp32 rounding)
 *   CLIPPED_RELU: min(max(y, 0), alpha)
 *   CLAMP:        min(max(y, alpha), beta)
 * followed, for int8 output, by the usual rounding and clip to [-128, 127]
 * (Relu keeps the TensorFlow form: clip to [0, 127]).  alpha and beta come
 * from fconv_plan_set_activation_params (default 0, 0). */
typedef enum {
  FCONV_ACT_NONE = 0,
  FCONV_ACT_RELU = 1,
  FCONV_ACT_LEAKY_RELU = 2,
  FCONV_ACT_CLIPPED_RELU = 3,
  FCONV_ACT_CLAMP = 4
} fconv_act;

/* Create a plan for one convolution shape.
 * N,H,W,C: input NHWC extents; K: output channels; R,S: filter height and
 * width; stride_h/stride_w >= 1; dilation is 1 and groups are 1 by
 * construction (the filter's input depth is C).
 * Constraints (else FCONV_ERR_NOT_SUPPORTED): C and K multiples of 16 for
 * int8 and of 8 for bf16 (16-byte vectors), and every tensor below 2^31
 * elements.  Non-positive extents, a VALID filter larger than
 * the input, or an unknown enum give FCONV_ERR_INVALID_VALUE.
 * Pure host work: needs no GPU.  *plan is set to NULL on failure. */
fconv_status fconv_plan_create(fconv_plan **plan, int N, int H, int W, int C,
                               int K, int R, int S, int stride_h, int stride_w,
                               fconv_padding padding, fconv_dtype dtype,
                               fconv_act act);

/* Parameters of the plan's activation: the slope for y < 0 (LEAKY_RELU), the
 * upper bound (CLIPPED_RELU, alpha >= 0), or the interval [alpha, beta]
 * (CLAMP, alpha <= beta); ignored by NONE and RELU.  Non-finite values or a
 * violated bound give FCONV_ERR_INVALID_VALUE and leave the plan unchanged.
 * Host only; applies to later runs. */
fconv_status fconv_plan_set_activation_params(fconv_plan *plan, float alpha,
                                              float beta);

/* Create a plan for a transposed convolution (the forward pass of a
 * deconvolution layer): "cudnn_deconvolution-inl.h" (MXNet), Forward, runs
 * cuDNN's backward-data pass of the cross-correlation with the op's pad and
 * stride and then adds the bias; here the bias and the rest of fconv_run's
 * epilogue are fused.  The sums are
 *   acc[n, p*sh + r - pad_top, q*sw + s - pad_left, k] += x[n, p, q, c] * w[r, s, c, k]
 * over input pixels p < H, q < W and taps whose target lies in the output,
 * which is Ho = (H-1)*sh + R - pad_top - pad_bottom by Wo (likewise).
 * MXNet's symmetric pad with output adjustment a is pad_top = pad,
 * pad_bottom = pad - a.  x: NHWC [N][H][W][C]; w: [R][S][C][K] (C input and
 * K output channels); y and side: [N][Ho][Wo][K].  Runs through every
 * fconv_run* entry point like any plan.  Strides up to 8, pads in
 * [0, filter-1] (the bottom/right pad down to 1 - stride, an output
 * adjustment larger than the pad), else FCONV_ERR_NOT_SUPPORTED; pads that
 * leave no output give FCONV_ERR_INVALID_VALUE.  Pure host work. */
fconv_status fconv_plan_create_transposed(fconv_plan **plan, int N, int H, int W,
                                          int C, int K, int R, int S,
                                          int stride_h, int stride_w,
                                          int pad_top, int pad_bottom,
                                          int pad_left, int pad_right,
                                          fconv_dtype dtype, fconv_act act);

/* Free a plan (NULL is accepted).  Does not synchronize any stream. */
fconv_status fconv_plan_destroy(fconv_plan *plan);

/* Output extents [N][P][Q][K]. */
fconv_status fconv_plan_output_shape(const fconv_plan *plan, int *N, int *P,
                                     int *Q, int *K);

/* Padding of the plan: top, bottom, left, right (for a transposed plan,
 * the pads it was created with). */
fconv_status fconv_plan_padding(const fconv_plan *plan, int *pad_top,
                                int *pad_bottom, int *pad_left,
                                int *pad_right);

/* Device scratch bytes fconv_run needs.  The TensorFlow GPU helper
 * ("conv_ops_fused_int8.cc", LaunchFusedConv2DOp for the GPU: the
 * DnnScratchAllocator and AllocateScratchOrFallback before the runner is
 * called) gives the fused convolution a scratch buffer of the size the
 * chosen algorithm asks for; here the caller allocates it, of this size,
 * and passes it to every run.  It holds a 16-bit copy of the filter in its
 * HWIO order for int8 plans (widened to fp16) and transposed plans (the
 * flipped taps; one per phase of a strided transposed plan) -- a bf16
 * forward plan reads the caller's filter as it is -- a 16-bit copy of the
 * input for int8 plans (only the strided pixels for a 1x1 strided plan)
 * and for transposed plans with a stride above the filter (zeros
 * inserted), and for a split-K plan (fconv_plan_set_splits) every unit's
 * 32-bit partial sums and one counter per tile and epilogue warp.  It
 * depends on the tile, split and gather in force: query it after changing
 * them.  It may be 0 (an unsplit bf16 forward plan, or a plan on the halo
 * gather, fconv_plan_set_gather); the run then accepts a NULL workspace. */
fconv_status fconv_workspace_size(const fconv_plan *plan, size_t *bytes);

/* Run the fused convolution on `stream`.
 * x, w, y: device pointers, 16-byte aligned.  bias: device fp32 [K].
 * side: device, output shape and dtype, 16-byte aligned, or NULL.
 * conv_scale, side_scale: host scalars (the TensorFlow GPU helper reads
 * them as host scalars too).  workspace: device, 256-byte aligned,
 * workspace_bytes >= fconv_workspace_size().  x/w must not alias y or
 * the workspace.  Asynchronous; returns after enqueueing.  A run is a
 * prep launch (the filter and input copies, split-K counters) and the
 * convolution launch, or the convolution alone for an unsplit bf16 forward
 * plan (fconv_plan_launch_count).  After a prep launch the convolution is
 * a programmatic dependent of it, which lets it start its set-up while the
 * prep finishes; it reads nothing the prep writes before that grid has
 * completed, and ordering against the caller's other work on the stream
 * is that of plain launches. */
fconv_status fconv_run(fconv_plan *plan, const void *x, const void *w,
                       const float *bias, const void *side, float conv_scale,
                       float side_scale, void *y, void *workspace,
                       size_t workspace_bytes, fconv_stream_t stream);

/* fconv_run with a per-output-channel conv_input_scale.
 * "conv_ops_fused_int8.cc" (TensorFlow), BiasActivationOutputKernel, step
 * (1) Scale: when the conv_input_scale tensor holds more than one element,
 * output channel k is scaled by its k-th element; otherwise by the scalar.
 * conv_scale: device fp32 [K], 16-byte aligned, read-only; y[..., k] is
 * computed with conv_scale[k] in step (1), every other step as in
 * fconv_run.  NULL conv_scale gives FCONV_ERR_INVALID_VALUE, a misaligned
 * one FCONV_ERR_MISALIGNED.  Same ownership, workspace and stream rules as
 * fconv_run. */
fconv_status fconv_run_channel_scale(fconv_plan *plan, const void *x,
                                     const void *w, const float *bias,
                                     const void *side, const float *conv_scale,
                                     float side_scale, void *y, void *workspace,
                                     size_t workspace_bytes,
                                     fconv_stream_t stream);

/* The convolution sums alone, before the epilogue: int32 [N][P][Q][K] for
 * int8 plans (exact), fp32 for bf16 plans.  Same rules as fconv_run. */
fconv_status fconv_run_accumulators(fconv_plan *plan, const void *x,
                                    const void *w, void *acc, void *workspace,
                                    size_t workspace_bytes,
                                    fconv_stream_t stream);

/* Batch-norm inference folded into fconv_run_channel_scale's arguments.
 * "use-fusion-api" (MIOpen), fusion plans: BatchNorm inference is one of
 * the fusable operators and the convolution-bias-batchnorm-activation
 * (CBNA) combination is listed for inference; the page gives no formula.
 * Read as the usual per-channel ("spatial") inference form applied to the
 * biased conv output, y_k -> gamma_k * (y_k - mean_k) / sqrt(var_k + eps)
 * + beta_k, which on y_k = acc * conv_scale + bias_k is again an affine map
 * of acc:
 *   g_k       = gamma_k / sqrt(var_k + eps)
 *   scale_out = conv_scale * g_k
 *   bias_out  = (bias_k - mean_k) * g_k + beta_k
 * each computed in double and rounded once to float.  A side input keeps
 * its own scale and is added after the normalisation (the residual add of
 * a conv-BN-add-Relu block).  All arrays are HOST fp32 [K] and are only
 * read (bias may be NULL: zero); scale_out and bias_out receive K values
 * each, for fconv_run_channel_scale's conv_scale and bias (after copying
 * them to the device).  FCONV_ERR_INVALID_VALUE for K <= 0, a NULL
 * required pointer, a non-finite or negative eps, or var_k + eps <= 0. */
fconv_status fconv_fold_batchnorm(int K, float conv_scale, const float *bias,
                                  const float *gamma, const float *beta,
                                  const float *mean, const float *var, float eps,
                                  float *scale_out, float *bias_out);

/* ---- Library-side entry points and controls.  The pages have no
 * counterpart for these: they run the operation above on host buffers,
 * expose and override this implementation's choices (tiles, chunking,
 * wait limits), and give tests their hooks. */

/* Bytes of device memory fconv_run_host needs: the workspace plus device
 * copies of x, w, bias, side (if with_side) and y. */
fconv_status fconv_host_workspace_size(const fconv_plan *plan, int with_side,
                                       size_t *bytes);

/* fconv_run on HOST buffers: copies x, w, bias and side (if not NULL) to
 * `device_workspace`, runs, and copies y back to `y_host`.  Large batches
 * are processed in chunks of images on two internal copy streams, so the
 * copy-in of one chunk and the copy-out of another overlap the compute of a
 * third (see fconv_plan_set_host_chunks); everything is ordered after the
 * work already queued on `stream`, and `stream` waits for the last copy-out.
 * Pinned host buffers keep this asynchronous; the caller synchronizes the
 * stream before reading y_host.  Pageable buffers work but make the copies
 * synchronous with the host.  A plan must not run two fconv_run_host calls
 * at once (they share its internal streams). */
fconv_status fconv_run_host(fconv_plan *plan, const void *x_host,
                            const void *w_host, const float *bias_host,
                            const void *side_host, float conv_scale,
                            float side_scale, void *y_host,
                            void *device_workspace, size_t workspace_bytes,
                            fconv_stream_t stream);

/* Number of batch chunks fconv_run_host pipelines over, split evenly
 * (1..16), or 0 for the automatic choice.  Automatic: a batch of at least
 * ten waves of output tiles (one tile per SM; u images a wave) takes chunks
 * of about u/6, u/2, 2u images, then middle chunks of about 3u, then 2u, u,
 * u/3, u/3, so that little of the copy-in, compute and copy-out is left
 * outside the overlap at either end; a smaller batch takes even chunks of
 * at least one wave each, at most 12, and one chunk when it has less. */
fconv_status fconv_plan_set_host_chunks(fconv_plan *plan, int chunks);

/* The image counts of the chunks fconv_run_host would use on a device with
 * `sm_count` SMs, in batch order (they sum to N): *count gets how many
 * (at most 16); `sizes`, when not NULL, gets them and must hold *count
 * entries (max_sizes), else FCONV_ERR_INVALID_VALUE.  Pure host work. */
fconv_status fconv_plan_host_chunk_sizes(const fconv_plan *plan, int sm_count,
                                         int *sizes, int max_sizes, int *count);

/* Status of the runs enqueued so far.  MIOpen's fusion API ("use-fusion-api",
 * running a fusion plan) reports an error for a run of a plan that cannot
 * execute; the kernels here run asynchronously, so a failure inside them
 * (a pipeline wait that ran out) is recorded on the device and read here.
 * Synchronizes `stream`, then reads and clears the current device's kernel
 * status word: FCONV_ERR_TIMEOUT if any kernel since the last check gave up
 * waiting, FCONV_ERR_CUDA if the stream reports an error, else FCONV_OK.
 * (fconv_run itself reports, before enqueueing anything, every error it can
 * see on the host: bad pointers, sizes and workspace.) */
fconv_status fconv_plan_check(fconv_plan *plan, fconv_stream_t stream);

/* Override the output-channel tile: 64, 128 or 256 (0 restores the
 * plan's own choice; K below the tile leaves zero columns).  int8 plans whose sums are chunked (more than 960
 * k-values) accept at most 128.  For benchmarking and tests. */
fconv_status fconv_plan_set_tile(fconv_plan *plan, int block_n);

/* Override the tile with `pixels` output pixels (128 or 256) x `channels`
 * output channels.  256-pixel tiles (two 128-pixel halves sharing each
 * filter tile) exist on the TMA im2col gather for 64 or 128 channels; other
 * shapes give FCONV_ERR_NOT_SUPPORTED.  fconv_plan_set_tile(plan, 0)
 * restores the automatic choice.  Host only. */
fconv_status fconv_plan_set_tile_shape(fconv_plan *plan, int pixels, int channels);

/* The plan's kernel configuration: output-channel tile, k-blocks summed in
 * one fp32 accumulator before they are folded into int32 (int8 plans), and
 * the number of output tiles. */
fconv_status fconv_plan_get_config(const fconv_plan *plan, int *block_n,
                                   int *kblocks_per_chunk, int *num_tiles);

/* Limit, in milliseconds, on any single pipeline wait inside the kernel
 * (default 2000).  After it the kernel stops, records FCONV_ERR_TIMEOUT and
 * returns. */
fconv_status fconv_plan_set_timeout_ms(fconv_plan *plan, uint32_t ms);

/* Test hooks.  FCONV_DEBUG_DROP_ARRIVE makes the input loaders skip their
 * "stage full" signal, so the MMA issuer's wait runs out and the kernel
 * exercises its timeout exit.  FCONV_DEBUG_GATHER_CPASYNC makes plans whose
 * channel count allows the TMA im2col input gather (C % 64 == 0) use the
 * general cp.async gather instead.  FCONV_DEBUG_ONE_KBLOCK_STAGES keeps
 * every pipeline stage at one k-block (plans that would fill two a stage,
 * "tma-im2col-kb2", run "tma-im2col").  FCONV_DEBUG_ONE_MMA_ISSUER keeps
 * one MMA-issuing thread and one accumulator on tiles that would split each
 * k-block's MMAs between two ("...-dual" kernels).  0 restores normal runs. */
#define FCONV_DEBUG_DROP_ARRIVE 1
#define FCONV_DEBUG_GATHER_CPASYNC 2
#define FCONV_DEBUG_ONE_KBLOCK_STAGES 4
#define FCONV_DEBUG_ONE_MMA_ISSUER 8
fconv_status fconv_plan_set_debug(fconv_plan *plan, int flags);

/* Record caller-created CUDA events (cudaEvent_t) at the stage boundaries
 * of every later fconv_run / fconv_run_accumulators on this plan, on the
 * run's stream: events[0] before the operand preparation (the filter copy
 * and, for int8 plans, the int8 -> fp16 input widening, one launch; none
 * for an unsplit bf16 forward plan), events[1] after it, events[2] before
 * the convolution kernel (the same point as events[1]), events[3] after
 * the convolution kernel.  For a strided
 * transposed plan events[1] and [2] follow the first phase's preparation
 * and events[3] the join of all phases.  NULL disables.  The events must
 * outlive the runs that record them. */
fconv_status fconv_plan_set_stage_events(fconv_plan *plan, void *const events[4]);

/* fconv_run for callers that cannot allocate device memory: a plugin inside
 * an engine that owns the whole device-memory budget, a latency-bound loop
 * where cudaMalloc/cudaFree (which can synchronize the device) is not
 * acceptable, or code limited to memory reserved at start-up.  The pages
 * have no counterpart of this call; it is a property of this library.
 * Same arguments and results as fconv_run, minus the workspace: the scratch
 * comes from a 32 MiB array the library reserves on every device that loads
 * it (held until the process exits).  Plans whose fconv_workspace_size()
 * exceeds 32 MiB get FCONV_ERR_WORKSPACE.  The call allocates nothing: no
 * cudaMalloc, cudaFree or allocating library routine.
 * The first call on each device looks up the array's device address (a
 * one-time set-up with that device current, repeated after cudaDeviceReset
 * gives the device a new context); make that first call before any stream
 * capture.  All calls on a device share the array and it keeps
 * the previous call's contents; each call writes every scratch byte it
 * reads, so nothing needs clearing, but calls whose kernels overlap on the
 * GPU (other streams, other host threads) race on it: serialize them. */
fconv_status fconv_run_no_alloc(fconv_plan *plan, const void *x, const void *w,
                                const float *bias, const void *side,
                                float conv_scale, float side_scale, void *y,
                                fconv_stream_t stream);

/* Where an int8 plan widens its activations to fp16 for the tensor cores.
 * FCONV_WIDEN_IN_KERNEL: inside the convolution kernel, from the int8 input
 * itself (no fp16 copy in the workspace), wherever the plan's tile allows it
 * (forward plans on the TMA im2col gather, C % 64 == 0, unsplit, 128-pixel
 * tiles of up to 128 channels or 256-pixel tiles of 64), else in the prep
 * launch; FCONV_WIDEN_COPY and FCONV_WIDEN_AUTO (the default, measured the
 * faster of the two on GB300): in the prep launch, into an fp16 copy of the
 * input in the workspace.  The workspace size depends on it
 * (query fconv_workspace_size after setting it); results do not.
 * fconv_plan_get_input_widening reports whether the next run widens inside
 * the kernel (1) or copies (0).  bf16 plans have nothing to widen. */
#define FCONV_WIDEN_AUTO 0
#define FCONV_WIDEN_IN_KERNEL 1
#define FCONV_WIDEN_COPY 2
fconv_status fconv_plan_set_input_widening(fconv_plan *plan, int mode);
fconv_status fconv_plan_get_input_widening(const fconv_plan *plan, int *in_kernel);

/* How the convolution kernel gathers its input operand.  The halo gather
 * serves forward stride-1 plans with C == 64 (or C == 32, int8), at most 9
 * filter taps, sums in one exact accumulation and 64-channel tiles, whose
 * input windows fit
 * shared memory (3x3 int8 layers up to 115 output columns, 86 on 256-pixel
 * tiles).
 * A tile is floor(128 * m / (Q + S - 1)) whole output rows of one image (m
 * = 1 or 2 for 128- or 256-pixel tiles), its GEMM rows those rows padded to
 * Q + S - 1 columns (the extra rows are computed and dropped).  Once a tile,
 * one tiled TMA copy brings the window of input rows the tile reads (zero
 * outside the image); the CTA's filter tile stays in shared memory, and the
 * MMA reads each filter tap's operand as a row shift of the window.  int8
 * plans widen the window and the filter inside the kernel: one launch, no
 * workspace (fconv_plan_set_input_widening with FCONV_WIDEN_COPY moves a
 * plan off this gather).  FCONV_GATHER_AUTO: the plan's own choice (the
 * default); FCONV_GATHER_IM2COL: never the halo gather; FCONV_GATHER_HALO:
 * the halo gather (FCONV_ERR_NOT_SUPPORTED for a plan it does not fit);
 * after it, fconv_plan_set_tile_shape(plan, 128 or 256, 64) picks the halo
 * tile of that height, while other tiles, fconv_plan_set_tile and split-K
 * are tiles of the other gathers.  The workspace size, launch count and tile
 * count depend on it; results do not (int8 bit for bit).
 * fconv_plan_kernel reports "tma-halo" / "tma-halo-m256". */
#define FCONV_GATHER_AUTO 0
#define FCONV_GATHER_IM2COL 1
#define FCONV_GATHER_HALO 2
fconv_status fconv_plan_set_gather(fconv_plan *plan, int mode);

/* Split-K for the plan's current tile: each output tile's k-blocks are
 * divided over `splits` CTAs (1: none; 0: the automatic choice made at
 * plan creation, tile included); every unit writes its partial sums to the
 * workspace and the last of a tile's units to finish adds them in split
 * order (int32 sums exactly, fp32 sums in that fixed order) and runs the
 * epilogue, so no CTA waits on another.  Forward plans on the TMA im2col
 * gather with 128-pixel tiles only (FCONV_ERR_NOT_SUPPORTED otherwise, and
 * for more splits than the plan has k-blocks); at most 8.  fconv_plan_set_tile and
 * fconv_plan_set_tile_shape reset it to 1.  The workspace size changes with
 * it: query fconv_workspace_size after setting it. */
fconv_status fconv_plan_set_splits(fconv_plan *plan, int splits);
fconv_status fconv_plan_get_splits(const fconv_plan *plan, int *splits);

/* Number of kernel launches one fconv_run (or fconv_run_channel_scale,
 * fconv_run_accumulators) on this plan enqueues: the operand preparation
 * (none for an unsplit bf16 forward plan) and the convolution, per phase
 * for a strided transposed plan, plus a small widening launch for int8
 * inputs whose size is not a multiple of 64. */
fconv_status fconv_plan_launch_count(const fconv_plan *plan, int *launches);

/* Which convolution kernel the plan's next run uses: "tma-im2col" (A
 * gathered by TMA im2col loads, 128-pixel tiles), "tma-im2col-kb2" (the
 * same with two k-blocks a pipeline stage: unsplit, unchunked tiles of up to
 * 128 channels and 12 or more k-blocks of 64), either with "-dual" (unsplit
 * tiles of up to 128 channels and 12 or more k-blocks: two threads issue
 * each k-block's MMAs into two accumulators the epilogue adds),
 * "tma-im2col-m256" (256-pixel tiles), "tma-halo" / "tma-halo-m256" (the
 * halo gather, fconv_plan_set_gather) or "cp-async" (the
 * general gather); for a strided transposed plan, its first phase's.
 * Static text; "" for a NULL plan. */
const char *fconv_plan_kernel(const fconv_plan *plan);

/* Static text for a status code. */
const char *fconv_status_string(fconv_status status);

/* Detail of the last failing call on this host thread ("" if none). */
const char *fconv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FCONV_H_ */
