// Host side of the fconv C ABI: plan creation (validation, output
// geometry, tile choice), workspace layout, tensor-map encoding and the
// launch sequence of one fused convolution.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <limits>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "fconv.h"
#include "fconv_internal.h"

struct fconv_plan {
  int N, H, W, C, K, R, S, sh, sw;
  fconv_padding padding;
  fconv_dtype dtype;
  fconv_act act;
  int P, Q, pt, pb, pl, pr;
  long long M;
  int Ktot, num_kb;
  int block_n, kb_chunk, num_n_tiles, num_tiles;
  int m_sub;            // 128-pixel sub-tiles per output tile (1 or 2)
  int splits;           // split-K units per tile (1: none; TMA gather only)
  int auto_splits;
  int auto_block_n, auto_m_sub;  // the automatic tile (and auto_splits)
  // the halo gather (fconv::Gather::kTmaHalo): whether the tile uses it, the
  // automatic choice, the caller's FCONV_GATHER_* mode, and its window
  int halo, auto_halo, gather_mode;
  int halo_q, halo_tr, halo_rows, tiles_per_img, halo_slot, halo_stg;
  uint32_t timeout_ms;
  int debug;
  size_t wt_bytes, xh_bytes;
  // int8 1x1 filter with a stride above 1: only the pixels the convolution
  // reads are widened, into a compact [N][P][Q][C] copy read at stride 1
  int subsample;
  // int8 activations widened inside the convolution kernel (no fp16 copy
  // of the input): widen_mode is the caller's choice (FCONV_WIDEN_*), widen
  // whether the next run does it (see update_widen)
  int widen_mode, widen;
  // the B tiles come from a 16-bit copy of the filter in the workspace
  // (int8 plans: widened; transposed plans: flipped taps) written by the
  // prep launch; otherwise (bf16 forward plans) straight from the caller's
  // HWIO filter
  int pack_filter;
  // transposed convolution: the filter is packed flipped in both spatial axes
  int transposed;
  // transposed convolution with a stride above the filter: the prep launch
  // copies x with stride-1 zero rows/columns inserted ((H-1)*sh+1 x
  // (W-1)*sw+1), and the convolution runs at stride 1 on that copy
  int upsample;
  int tpad[4];   // a transposed plan's pads as given (top, bottom, left, right)
  // the filter copy's taps (see fconv::WidenMap); tap_nR == 0: as given
  int tap_nR, tap_nS, tap_R, tap_S, tap_r0, tap_s0, tap_rstep, tap_sstep;
  // output pixel map (see fconv::ConvArgs); omap == 0: GEMM row = pixel
  int omap, out_H, out_W, o_sh, o_sw, o_h0, o_w0;
  // where this plan's filter copy and input copy sit in the workspace
  size_t ws_wt_off, ws_xh_off;
  // a strided transposed convolution runs as sh*sw phases, each a forward
  // plan over x with every stride-th filter tap, writing every stride-th
  // output row and column (owned by this plan)
  int num_phases;
  fconv_plan *phase[64];
  int sm_share;   // a phase: how many phases share the SMs at once (tile choice)
  // side streams on which the phases after the first run concurrently with
  // it (fork after the input copy, join before the run returns)
  int fork_dev;   // device they belong to, -1 = none
  int num_fork;
  cudaStream_t fork_s[3];
  cudaEvent_t fork_start, fork_done[3];
  float act_alpha, act_beta;   // activation parameters (fconv_plan_set_activation_params)
  cudaEvent_t events[4];
  bool use_events;
  // fconv_run_host pipeline: batch chunks, two copy streams and their events
  int host_chunks;  // 0 = automatic
  int pipe_dev;     // device the streams/events below belong to, -1 = none
  cudaStream_t s_in, s_out;
  cudaEvent_t ev_entry, ev_out, ev_in[16], ev_comp[16];
  // tensor maps of the last run, reused while what they encode is unchanged
  // (the tensor's address, the batch size, the tile)
  struct MapCache {
    bool valid;
    const void *base;
    int n, form;   // A: batch size, and 1 for the int8 input itself (widening)
    CUtensorMap map;
  } map_a, map_b;
};

constexpr int kMaxHostChunks = 16;

namespace {

thread_local std::string t_last_error;

fconv_status fail(fconv_status st, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return st;
}

fconv_status cuda_fail(cudaError_t e, const char *what) {
  return fail(FCONV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
constexpr long long kLimit = 0x7FFFFFFFLL;
// split-K: at most this many units per tile, each of at least
// kMinSplitKBlocks k-blocks; one completion counter per tile and TMA
// epilogue warp
constexpr int kMaxSplits = 8;
constexpr int kMinSplitKBlocks = 4;
constexpr int kSplitCountersPerTile = 8;

// Output extent and padding split of one axis under TensorFlow's rule:
// SAME keeps ceil(in / stride) outputs and pads max(0, (out-1)*stride +
// filt - in) in total, the smaller half before; VALID pads nothing.
bool axis_geometry(int in, int filt, int stride, fconv_padding pad, int *out, int *before,
                   int *after) {
  if (pad == FCONV_VALID) {
    if (filt > in) return false;
    *out = (in - filt) / stride + 1;
    *before = *after = 0;
    return true;
  }
  const int o = (in + stride - 1) / stride;
  long long total = static_cast<long long>(o - 1) * stride + filt - in;
  if (total < 0) total = 0;
  *out = o;
  *before = static_cast<int>(total / 2);
  *after = static_cast<int>(total - total / 2);
  return true;
}

int sm_count_of_current_device(int fallback) {
  int dev = 0, v = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();  // clear the non-sticky error of a GPU-less host
    return fallback;
  }
  return v;
}

// The input as the convolution kernels read it: extents and strides.
struct InputView {
  int H, W, sh, sw;
};
InputView input_view(const fconv_plan &p) {
  if (p.widen) return {p.H, p.W, p.sh, p.sw};  // the int8 input itself
  if (p.subsample) return {p.P, p.Q, 1, 1};   // compact copy of the strided pixels
  if (p.upsample) return {(p.H - 1) * p.sh + 1, (p.W - 1) * p.sw + 1, 1, 1};
  return {p.H, p.W, p.sh, p.sw};
}

// The A tile can be loaded by one TMA im2col copy when a k-block never
// straddles two filter taps (C % 64 == 0) and the convolution fits the
// tensor map's limits for a 4-D tensor: bounding-box corners in [-128, 127],
// traversal strides <= 8, filter offsets small.
bool im2col_ok(const fconv_plan &p) {
  const InputView v = input_view(p);
  const int sh = v.sh, sw = v.sw;
  if (p.pt < 0 || p.pl < 0) return false;   // window origins starting inside the image
  if (p.C % 64 != 0 || sh > 8 || sw > 8 || p.R > 16 || p.S > 16) return false;
  const int corners[4] = {-p.pl, -p.pt, p.pr - (p.S - 1), p.pb - (p.R - 1)};
  for (int c : corners)
    if (c < -128 || c > 127) return false;
  return true;
}

// The gather a run uses for a given tile: TMA im2col when the shape and
// tile allow it, else the general cp.async gather.
fconv::Gather gather_for(const fconv_plan &p, int bn, bool force_cpasync) {
  const bool chunked = p.kb_chunk < p.num_kb;
  if (!force_cpasync && im2col_ok(p) && fconv::gather_supports(fconv::Gather::kTmaIm2col, bn, chunked))
    return fconv::Gather::kTmaIm2col;
  return fconv::Gather::kCpAsync;
}

// Whether the next run uses the halo gather (the cp.async test hook wins).
bool halo_run(const fconv_plan &p) {
  return p.halo && !(p.debug & FCONV_DEBUG_GATHER_CPASYNC);
}

// The gather the next run of a plan uses.
fconv::Gather gather_for_run(const fconv_plan &p) {
  if (halo_run(p)) return fconv::Gather::kTmaHalo;
  return gather_for(p, p.block_n, (p.debug & FCONV_DEBUG_GATHER_CPASYNC) != 0);
}

// The halo gather's tiles of 128 * ms GEMM rows x 64 channels, and
// whether the plan can use them: a forward stride-1 plan with C == 64 (one
// k-block a filter tap) whose sums fit one fp32 accumulation, whose filter
// tile (R * S blocks of 64 x 64, 8 KB each) stays resident and whose input
// window fits its buffer.  A tile is tr = floor(128 * ms / q) whole output
// rows padded to q = Q + S - 1 columns (an image takes ceil(P / tr) tiles);
// its window is tr + R - 1 input rows of q pixels.  Shared memory holds two
// 16-bit windows, for int8 two stagings of the int8 window (each window is
// copied while the previous one is widened), and the filter tile.  An int8
// window is widened inside the kernel, so a plan that asks for the fp16
// input copy (FCONV_WIDEN_COPY) does not use the gather.
struct HaloGeom {
  int q, tr, rows, tiles_per_img, slot, stg;
};
bool halo_geometry(const fconv_plan &p, int ms, HaloGeom *g) {
  if (p.transposed || p.upsample || p.subsample || p.tap_nR > 0 || p.num_phases > 0) return false;
  // C == 32 (int8): a window pixel's upper 32 channels are the copy's zero
  // fill and the filter tile's rows for them zero
  const bool c_ok = p.C == 64 || (p.C == 32 && p.dtype == FCONV_INT8);
  if (p.sh != 1 || p.sw != 1 || !c_ok || p.pt < 0 || p.pl < 0) return false;
  const int taps = p.R * p.S;
  if (p.kb_chunk < p.num_kb || taps * 64 * 64 * 2 > fconv::kHaloBMax) return false;
  if (p.dtype == FCONV_INT8 && p.widen_mode == FCONV_WIDEN_COPY) return false;
  if (ms != 1 && ms != 2) return false;
  const int q = p.Q + p.S - 1;
  if (q > 128 * ms || q > 256) return false;
  const int tr = 128 * ms / q;
  const int rows = tr + p.R - 1;
  if (rows > 256) return false;
  const long long px = static_cast<long long>(rows) * q;
  const long long slot = (px * 128 + 1023) / 1024 * 1024;
  const long long stg = p.dtype == FCONV_INT8 ? (px * 64 + 511) / 512 * 512 : 0;
  if (2 * slot + 2 * stg + taps * 64LL * 64 * 2 > fconv::kHaloRegion) return false;
  const long long tpi = (p.P + tr - 1) / tr;
  if (tpi * p.N * ((p.K + 63) / 64) > kLimit) return false;
  // every CTA keeps one channel tile: at least one CTA for each of them
  if ((p.K + 63) / 64 > sm_count_of_current_device(148)) return false;
  if (g) *g = {q, tr, rows, static_cast<int>(tpi), static_cast<int>(slot), static_cast<int>(stg)};
  return true;
}

// K-blocks a pipeline stage of the next run: 2 on the TMA gather for
// unsplit, unchunked 128-pixel tiles of up to 128 channels and at least
// kKps2MinKBlocks k-blocks, without in-kernel widening (a producer fills at
// most one stage per ~550-650 cycles, so larger stages halve its cost per
// k-block; on tiles of a few k-blocks the ring's coarser stages measured
// slower: 64x28x28x256 1x1, 4 k-blocks, 33.5 -> 35.0 us a graph step),
// else 1.
constexpr int kKps2MinKBlocks = 12;
int kblocks_per_stage(const fconv_plan &p) {
  if (p.debug & FCONV_DEBUG_ONE_KBLOCK_STAGES) return 1;
  const bool ok = gather_for_run(p) == fconv::Gather::kTmaIm2col && p.m_sub == 1 &&
                  p.block_n <= 128 && p.splits == 1 && !p.widen && p.kb_chunk >= p.num_kb &&
                  p.num_kb >= kKps2MinKBlocks;
  return ok ? 2 : 1;
}

// Whether the next run splits each k-block's MMAs between two issuing
// threads (two accumulators, added in the epilogue): the TMA gather's
// unsplit 128-pixel tiles of up to 128 channels with at least
// kKps2MinKBlocks k-blocks, where one thread's MMA issue (~110 cycles an
// MMA, 4 a k-block) bounds the mainloop; short tiles keep one accumulator,
// whose epilogue reads half as much tensor memory.
bool split_mma_issue(const fconv_plan &p) {
  if (p.debug & FCONV_DEBUG_ONE_MMA_ISSUER) return false;
  return gather_for_run(p) == fconv::Gather::kTmaIm2col && p.m_sub == 1 && p.block_n <= 128 &&
         p.splits == 1 && !p.widen && p.num_kb >= kKps2MinKBlocks;
}


// Tile: the candidate (BN output channels x 128*MS output pixels) with the
// least estimated time.  A unit (a tile, or its split) costs the longer of
// its mainloop and its epilogue, which runs while the next unit's mainloop
// does.  A k-block costs about max(2*BN*MS, G) cycles: the
// MMAs of a 128 x BN x 64 block take ~2*BN on the tensor core, and the
// issuing threads' per-k-block work (barrier waits, copy and MMA issue) a
// fixed G whatever BN is (~500 on the TMA path with one 128-pixel sub-tile,
// ~700 with two and two MMA issuers, ~800 on the cp.async path; measured
// per k-block in steady state, operand traffic included).  Tiles run in waves
// over the SMs; the epilogue of a CTA's last tile (~8 cycles per output
// column per 128 pixels) is not hidden behind a next tile's mainloop.
// Split-K (splits > 1 units per tile, TMA gather, forward plans): a unit
// runs ceil(num_kb / splits) k-blocks; every unit writes its partial sums
// (128*MS x BN 32-bit words) and the last to finish reads all of them
// back, ~8 cycles per output column per 128 pixels per split at an SM's
// ~64 bytes per cycle from L2, before the epilogue.
struct TileChoice {
  int bn, ms, splits, halo;
};
TileChoice choose_tile(const fconv_plan &p, int sms, bool allow_halo = true) {
  const bool chunked = p.kb_chunk < p.num_kb;
  // runs with a prep launch whatever the split: an input copy or a filter copy
  const bool needs_prep = p.dtype == FCONV_INT8 || p.upsample || p.transposed;
  const int kp = (p.K + 63) / 64 * 64;   // tiles are whole 64-channel B boxes
  TileChoice best = {64, 1, 1, 0};
  long long best_cost = -1;
  // the halo gather (64-channel tiles, unsplit): per k-block each MMA
  // issuer's 4 MMAs (~110 cycles each, two issuers on 256-pixel tiles)
  // against the tensor core's ~48 cycles a 128 x 64 x 16 MMA; the window
  // copy and widening run on other warps a tile ahead.  (The im2col tiles'
  // int8 input copy in the prep launch, which this gather avoids, is not
  // counted.)
  for (int ms : {1, 2}) {
    HaloGeom g;
    if (!allow_halo || !halo_geometry(p, ms, &g)) continue;
    const long long tiles = static_cast<long long>(p.N) * g.tiles_per_img * ((p.K + 63) / 64);
    const long long waves = (tiles + sms - 1) / sms;
    const long long mainloop = static_cast<long long>(p.R) * p.S * (192LL * ms > 440 ? 192LL * ms : 440);
    const long long epilogue = 22LL * 64 * ms;
    const long long cost = waves * (mainloop > epilogue ? mainloop : epilogue) + 8LL * 64 * ms;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = {64, ms, 1, 1};
    }
  }
  for (int bn : {256, 128, 64}) {
    for (int ms : {1, 2}) {
      if (bn > kp) continue;
      fconv::Gather g = gather_for(p, bn, false);
      if (!fconv::gather_supports(g, bn, chunked, ms)) continue;
      // 128-pixel tiles of <= 128 channels, unsplit and unchunked, run two
      // k-blocks a stage (costed as one MMA issuer: 4 MMAs of ~105 cycles a
      // k-block; they run with two, split_mma_issue, which measured faster
      // on the 32x14x14x256 bf16 layer, 14.3 -> 12.4 us a graph step, but
      // costing them so moved the bf16 4x4/2 transposed layer's phases to
      // 128 x 128 tiles, 30.5 -> 36.7 us)
      const bool kb2 = g == fconv::Gather::kTmaIm2col && ms == 1 && bn <= 128 && !chunked &&
                       p.num_kb >= 12;   // kblocks_per_stage's rule
      const long long fixed =
          g == fconv::Gather::kTmaIm2col ? (ms == 2 ? 700 : 500) : 800;
      const long long m_tiles = (p.M + 128LL * ms - 1) / (128LL * ms);
      const long long tiles = m_tiles * ((p.K + bn - 1) / bn);
      const long long work = 2LL * bn * ms;
      const bool can_split = g == fconv::Gather::kTmaIm2col && !p.transposed && ms == 1;
      for (int sp = 1; sp <= (can_split ? kMaxSplits : 1); ++sp) {
        if (sp > 1 && (tiles * sp > sms || p.num_kb < kMinSplitKBlocks * sp)) break;
        const long long units = tiles * sp;
        const long long waves = (units + sms - 1) / sms;
        const long long kbs = (p.num_kb + sp - 1) / sp;
        // a tile's epilogue overlaps the next tile's mainloop, so a unit
        // costs the longer of the two: ~1400 cycles per 32-column slice of
        // each epilogue warp (BN / 64 slices a warp, twice that with two
        // sub-tiles), i.e. ~22 * BN * MS
        const long long g_kb = (kb2 && sp == 1) ? 420 : fixed;
        const long long mainloop = kbs * (work > g_kb ? work : g_kb);
        const long long epilogue = 22LL * bn * ms;
        // split-K needs its counters zeroed by a prep launch; a plan with no
        // other prep work (bf16 forward) pays a whole launch for it (~4 us)
        const long long split_launch = (sp > 1 && !needs_prep) ? 8000 : 0;
        // an int8 run's prep launch (the fp16 input copy), which the halo
        // gather's candidates above do not have
        const long long prep_launch = (p.dtype == FCONV_INT8 && halo_geometry(p, 1, nullptr))
                                          ? 6000 : 0;
        const long long cost = waves * (mainloop > epilogue ? mainloop : epilogue) +
                               8LL * bn * ms + (sp > 1 ? 8LL * bn * ms * (sp + 1) : 0) +
                               split_launch + prep_launch;
        if (best_cost < 0 || cost < best_cost) {
          best_cost = cost;
          best = {bn, ms, sp, 0};
        }
      }
    }
  }
  return best;
}

void update_widen(fconv_plan &p);
void set_tiling(fconv_plan &p, int bn, int ms, int splits, int halo);

// Move a plan off the halo gather, onto the automatic tile without it.
void retile_without_halo(fconv_plan &p) {
  const int sms = sm_count_of_current_device(148);
  const TileChoice t = choose_tile(p, p.sm_share > 1 ? sms / p.sm_share : sms, false);
  set_tiling(p, t.bn, t.ms, t.splits, 0);
}

// Output tiles of the plan's tile shape (the halo gather tiles each image's
// virtual pixels).
int tile_count(const fconv_plan &p) {
  if (p.halo) return p.N * p.tiles_per_img * p.num_n_tiles;
  return static_cast<int>((p.M + 128LL * p.m_sub - 1) / (128LL * p.m_sub)) * p.num_n_tiles;
}

// halo: use the halo gather (the caller has checked halo_geometry).
void set_tiling(fconv_plan &p, int bn, int ms, int splits, int halo) {
  p.block_n = bn;
  p.m_sub = ms;
  HaloGeom g = {0, 0, 0, 0, 0, 0};
  p.halo = (halo && bn == 64 && splits <= 1 && halo_geometry(p, ms, &g)) ? 1 : 0;
  p.halo_q = g.q;
  p.halo_tr = g.tr;
  p.halo_rows = g.rows;
  p.tiles_per_img = g.tiles_per_img;
  p.halo_slot = g.slot;
  p.halo_stg = g.stg;
  // no empty unit: with ceil(num_kb / splits) k-blocks a unit, that many
  // units cover the tile (9 k-blocks asked in 4 splits run as 3 of 3)
  if (splits > 1) {
    const int per = (p.num_kb + splits - 1) / splits;
    splits = (p.num_kb + per - 1) / per;
  }
  p.splits = splits < 1 ? 1 : splits;
  p.num_n_tiles = (p.K + bn - 1) / bn;
  p.num_tiles = tile_count(p);
  update_widen(p);
}

// Whether int8 activations can be widened inside the convolution kernel
// under the plan's tile: a forward int8 plan on the TMA gather (judged on
// the input as it is), unsplit, with epilogue threads holding at most 64
// sums (128-pixel tiles of up to 128 channels, 256-pixel tiles of 64).
bool widen_eligible(const fconv_plan &p) {
  if (p.dtype != FCONV_INT8 || p.transposed || p.upsample || p.splits != 1 || p.halo) return false;
  if (p.debug & FCONV_DEBUG_GATHER_CPASYNC) return false;
  if (p.m_sub == 1 ? p.block_n > 128 : p.block_n != 64) return false;
  fconv_plan raw = p;
  raw.widen = 1;   // the input view of the raw input
  return im2col_ok(raw);
}

// The widening choice and the workspace it implies: with in-kernel
// widening there is no fp16 input copy.  FCONV_WIDEN_AUTO copies: measured
// on the int8 workloads (CUDA graphs, GB300), the prep launch's fp16 copy
// was faster wherever in-kernel widening applies (32x56x56x64 3x3 22.5 us
// against 38.8; 64x28x28x256 1x1 34.0 against 43.1; the 1x1 stride-2 layer
// 17.2 against 18.4): the two converter warps bound the mainloop and share
// the SM with the epilogue, while HBM has room for the copy.
void update_widen(fconv_plan &p) {
  const bool want = p.widen_mode == FCONV_WIDEN_IN_KERNEL;
  p.widen = (want && widen_eligible(p)) ? 1 : 0;
  const InputView v = input_view(p);
  const long long xh_elems = static_cast<long long>(p.N) * v.H * v.W * p.C;
  p.xh_bytes = ((p.dtype == FCONV_INT8 && !p.widen && !halo_run(p)) || p.upsample)
                   ? align_up(static_cast<size_t>(xh_elems) * 2, 256) : 0;
}

PFN_cuTensorMapEncodeIm2col_v12000 encode_im2col_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeIm2col_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

struct DeviceInfo {
  std::atomic<int> sm_count{0};
};
DeviceInfo g_devices[64];

int device_sm_count(int *dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (dev_out) *dev_out = dev;
  if (dev < 0 || dev >= 64) return sm_count_of_current_device(-1);
  int v = g_devices[dev].sm_count.load();
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_devices[dev].sm_count.store(v);
  }
  return v;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


// Scratch a run needs: the filter copy, and for int8 plans the fp16 copy of
// the input the gathers read.
// Split-K scratch after the operand copies: every unit's partial block
// (128 * m_sub * block_n 32-bit words), then one counter per tile and
// epilogue warp.
// Bytes of the filter copy a run writes (an int8 plan on the halo gather
// widens its filter inside the convolution kernel instead).
size_t filter_copy_bytes(const fconv_plan &p) {
  return (p.pack_filter && !(halo_run(p) && p.dtype == FCONV_INT8)) ? p.wt_bytes : 0;
}
// End of the operand copies in the workspace.
size_t copies_end(const fconv_plan &p) {
  const size_t wt = filter_copy_bytes(p);
  const size_t a = wt ? p.ws_wt_off + wt : 0, b = p.xh_bytes ? p.ws_xh_off + p.xh_bytes : 0;
  return a > b ? a : b;
}
size_t split_partial_offset(const fconv_plan &p) {
  return align_up(copies_end(p), 256);
}
size_t split_partial_bytes(const fconv_plan &p) {
  return align_up(static_cast<size_t>(p.num_tiles) * p.splits * 128 * p.m_sub * p.block_n * 4, 256);
}
size_t workspace_need(const fconv_plan &p) {
  if (p.splits > 1)
    return split_partial_offset(p) + split_partial_bytes(p) +
           align_up(static_cast<size_t>(p.num_tiles) * kSplitCountersPerTile * 4, 256);
  return copies_end(p);
}

fconv_plan batch_slice(const fconv_plan &p, int n);
fconv_status ensure_fork(fconv_plan *p);

fconv_status enqueue(fconv_plan *p, const void *x, const void *w, const float *bias,
                     const void *side, float conv_scale, float side_scale, void *y,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream, int mode,
                     bool skip_pack = false, const float *scale_k = nullptr,
                     bool skip_copy = false, bool prep_only = false) {
  if (!p) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (!x || !w || !y) return fail(FCONV_ERR_INVALID_VALUE, "x, w and y must not be NULL");
  if (mode == fconv::kModeFused && !bias)
    return fail(FCONV_ERR_INVALID_VALUE, "bias must not be NULL");
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || (side && !aligned(side, 16)) ||
      (bias && !aligned(bias, 16)) || (scale_k && !aligned(scale_k, 16)))
    return fail(FCONV_ERR_MISALIGNED,
                "x, w, y, side, bias and the per-channel scale must be 16-byte aligned");
  const size_t need = workspace_need(*p);
  if (need > 0 && (!workspace || workspace_bytes < need))
    return fail(FCONV_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need,
                workspace ? workspace_bytes : static_cast<size_t>(0));
  if (workspace && !aligned(workspace, 256))
    return fail(FCONV_ERR_MISALIGNED, "workspace must be 256-byte aligned");

  int dev = 0;
  const int sms = device_sm_count(&dev);
  if (sms <= 0) return fail(FCONV_ERR_CUDA, "no usable CUDA device");
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn();
  if (!encode) return fail(FCONV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");

  const bool is_int8 = p->dtype == FCONV_INT8;
  auto mark = [&](int i) -> cudaError_t {
    return p->use_events ? cudaEventRecord(p->events[i], stream) : cudaSuccess;
  };
  uint16_t *wt = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) + p->ws_wt_off);
  __half *xh = reinterpret_cast<__half *>(static_cast<uint8_t *>(workspace) + p->ws_xh_off);

  if (p->num_phases > 0) {
    // one forward plan per phase: the first one's prep (which also widens
    // the input, int8) on the caller's stream, then the other phases on
    // side streams concurrently with the first one's convolution
    fconv_status st = ensure_fork(p);
    if (st != FCONV_OK) return st;
    fconv_plan tmp[64];
    fconv_plan *q[64];
    for (int i = 0; i < p->num_phases; ++i) {
      q[i] = p->phase[i];
      if (q[i]->N != p->N) {
        tmp[i] = batch_slice(*q[i], p->N);
        q[i] = &tmp[i];
      }
      q[i]->act = p->act;
      q[i]->act_alpha = p->act_alpha;
      q[i]->act_beta = p->act_beta;
      q[i]->debug = p->debug;
      q[i]->timeout_ms = p->timeout_ms;
    }
    cudaError_t e0 = mark(0);
    if (e0 != cudaSuccess) return cuda_fail(e0, "event record");
    st = enqueue(q[0], x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
                 stream, mode, skip_pack, scale_k, skip_copy, /*prep_only=*/true);
    if (st != FCONV_OK) return st;
    if ((e0 = mark(1)) != cudaSuccess || (e0 = mark(2)) != cudaSuccess)
      return cuda_fail(e0, "event record");
    const int nf = p->num_phases > 1 ? p->num_fork : 0;
    if (nf > 0) {
      if ((e0 = cudaEventRecord(p->fork_start, stream)) != cudaSuccess)
        return cuda_fail(e0, "event record");
      for (int j = 0; j < nf; ++j)
        if ((e0 = cudaStreamWaitEvent(p->fork_s[j], p->fork_start, 0)) != cudaSuccess)
          return cuda_fail(e0, "stream ordering");
    }
    for (int i = 1; i < p->num_phases; ++i) {
      st = enqueue(q[i], x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
                   p->fork_s[(i - 1) % nf], mode, skip_pack, scale_k, /*skip_copy=*/true);
      if (st != FCONV_OK) return st;
    }
    // the first phase's convolution (its operands are ready)
    st = enqueue(q[0], x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
                 stream, mode, /*skip_pack=*/true, scale_k, /*skip_copy=*/true);
    if (st != FCONV_OK) return st;
    for (int j = 0; j < nf; ++j)
      if ((e0 = cudaEventRecord(p->fork_done[j], p->fork_s[j])) != cudaSuccess ||
          (e0 = cudaStreamWaitEvent(stream, p->fork_done[j], 0)) != cudaSuccess)
        return cuda_fail(e0, "stream ordering");
    if ((e0 = mark(3)) != cudaSuccess) return cuda_fail(e0, "event record");
    return FCONV_OK;
  }

  const fconv::Gather gather = gather_for_run(*p);
  // two 128-pixel sub-tiles and split-K exist on the TMA gather only: a plan
  // forced onto the cp.async gather (a test hook) runs this launch with one
  // unsplit 128-pixel tile, from a copy, so the caller's plan keeps its
  // tiling (and its workspace size)
  fconv_plan reduced;
  if (gather == fconv::Gather::kCpAsync && (p->m_sub != 1 || p->splits != 1 || p->halo)) {
    reduced = *p;
    set_tiling(reduced, p->block_n, 1, 1, 0);
    p = &reduced;
  }
  if (!fconv::gather_supports(gather, p->block_n, p->kb_chunk < p->num_kb, p->m_sub))
    return fail(FCONV_ERR_NOT_SUPPORTED,
                "tile %d has no cp.async kernel for a sum of %d k-values (chunked sums need "
                "BN <= 128 there)", p->block_n, p->Ktot);

  cudaError_t e = mark(0);
  if (e != cudaSuccess) return cuda_fail(e, "event record");
  // filter copy (int8 widened; transposed plans' taps flipped) and input
  // copy (int8 widening; subsampled or upsampled copies) in one launch; the
  // convolution reads the copies when there are some
  const InputView view = input_view(*p);
  const int gH = view.H, gW = view.W, gsh = view.sh, gsw = view.sw;
  const bool halo = gather == fconv::Gather::kTmaHalo;
  // the convolution reads a copy (the halo gather widens int8 windows itself)
  const bool copy = (is_int8 && !p->widen && !halo) || p->upsample;
  const bool do_copy = copy && !skip_copy;            // ... made by this launch
  const void *act = x;
  const long long n = static_cast<long long>(p->N) * gH * gW * p->C;
  // split-K scratch: partial sums, then the completion counters (zeroed by
  // the prep launch of every run)
  uint32_t *split_partial = nullptr;
  int *split_counters = nullptr;
  if (p->splits > 1) {
    uint8_t *base = static_cast<uint8_t *>(workspace) + split_partial_offset(*p);
    split_partial = reinterpret_cast<uint32_t *>(base);
    split_counters = reinterpret_cast<int *>(base + split_partial_bytes(*p));
  }
  // (a run whose filter needs no copy, or has it already, and whose input
  // needs none either still launches it when split-K counters need zeroing)
  const bool do_pack = !skip_pack && filter_copy_bytes(*p) > 0;
  const bool prep = do_pack || do_copy || split_counters;
  if (prep) {
    fconv::WidenMap map;
    memset(&map, 0, sizeof map);
    map.mode = p->subsample ? fconv::kCopySubsample
                            : p->upsample ? fconv::kCopyUpsample : fconv::kCopyDense;
    map.C = p->C; map.H = p->H; map.W = p->W; map.P = gH; map.Q = gW;
    map.sh = p->sh; map.sw = p->sw;
    map.tap_nR = p->tap_nR; map.tap_nS = p->tap_nS; map.tap_R = p->tap_R; map.tap_S = p->tap_S;
    map.tap_r0 = p->tap_r0; map.tap_s0 = p->tap_s0;
    map.tap_rstep = p->tap_rstep; map.tap_sstep = p->tap_sstep;
    e = fconv::launch_prep(is_int8, do_pack ? w : nullptr, wt, p->Ktot, p->K, x, xh,
                           do_copy ? n : 0, map, split_counters,
                           split_counters ? p->num_tiles * kSplitCountersPerTile : 0, sms,
                           stream);
    if (e != cudaSuccess) return cuda_fail(e, "operand preparation launch");
  }
  if (copy) act = xh;
  if (prep_only) return FCONV_OK;
  if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "event record");
  if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "event record");

  // B: the filter as the [R*S*C][K] matrix of its HWIO layout, 16-bit, in
  // blocks of 64 output channels x 64 k-rows (rows past R*S*C and channels
  // past K read as zero).  K a multiple of 64 (and at least block_n): the
  // 3-D view {64 channels, rows, K / 64 blocks} (row stride K * 2 bytes,
  // block stride 128 bytes), whose {64, 64, block_n / 64} box is a whole B
  // tile in one copy; else the 2-D matrix in 64 x 64 boxes.
  const void *bsrc = p->pack_filter ? static_cast<const void *>(wt) : w;
  // an int8 plan on the halo gather reads the caller's int8 filter itself
  const bool b_map = !(halo && is_int8);
  const int b3d = (p->K % 64 == 0 && p->block_n <= p->K) ? 1 : 0;
  const int kps = kblocks_per_stage(*p);   // boxes of 64 * kps k-rows
  const int b_form = b3d | (kps << 1);
  fconv_plan::MapCache &mb = p->map_b;
  if (b_map &&
      !(mb.valid && mb.base == bsrc && mb.form == b_form && (!b3d || mb.n == p->block_n))) {
    mb.valid = false;
    memset(&mb.map, 0, sizeof mb.map);
    const CUtensorMapDataType bt =
        is_int8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult cr;
    if (b3d) {
      const cuuint64_t gdim[3] = {64, static_cast<cuuint64_t>(p->Ktot),
                                  static_cast<cuuint64_t>(p->K / 64)};
      const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(p->K) * 2, 128};
      const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(64 * kps),
                                 static_cast<cuuint32_t>(p->block_n / 64)};
      const cuuint32_t estride[3] = {1, 1, 1};
      cr = encode(&mb.map, bt, 3, const_cast<void *>(bsrc), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
      const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(p->K),
                                  static_cast<cuuint64_t>(p->Ktot)};
      const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(p->K) * 2};
      const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(64 * kps)};
      const cuuint32_t estride[2] = {1, 1};
      cr = encode(&mb.map, bt, 2, const_cast<void *>(bsrc), gdim, gstride, box, estride,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (cr != CUDA_SUCCESS)
      return fail(FCONV_ERR_INTERNAL, "tensor map encode failed (%d)", (int)cr);
    mb.base = bsrc;
    mb.n = p->block_n;
    mb.form = b_form;
    mb.valid = true;
  }
  static const CUtensorMap kNoMapB = {};
  const CUtensorMap &tmap = b_map ? mb.map : kNoMapB;

  // A: one im2col copy per k-block of a whole tile's pixels (128, or 256
  // for two sub-tiles: the second continues the first's walk); widening in
  // the kernel copies each 128-pixel sub-tile into its own staging slot
  const int a_pixels = p->widen ? 128 : 128 * p->m_sub;
  const int a_form = halo ? (3 | (p->halo_q << 2) | (p->halo_rows << 11))
                          : (p->widen ? 1 : 0) | (a_pixels << 2);
  fconv_plan::MapCache &ma = p->map_a;
  if (halo && !(ma.valid && ma.base == act && ma.n == p->N && ma.form == a_form)) {
    // the input itself, NHWC, innermost first: C, W, H, N; a box of the 64
    // channels of halo_rows x halo_q pixels (parts outside the image read
    // as zero); int8 unswizzled (the kernel widens it), bf16 with the
    // 128-byte swizzle the MMA reads
    ma.valid = false;
    memset(&ma.map, 0, sizeof ma.map);
    const int elt = is_int8 ? 1 : 2;
    const cuuint64_t hdim[4] = {static_cast<cuuint64_t>(p->C), static_cast<cuuint64_t>(p->W),
                                static_cast<cuuint64_t>(p->H), static_cast<cuuint64_t>(p->N)};
    const cuuint64_t hstride[3] = {static_cast<cuuint64_t>(p->C) * elt,
                                   static_cast<cuuint64_t>(p->W) * p->C * elt,
                                   static_cast<cuuint64_t>(p->H) * p->W * p->C * elt};
    const cuuint32_t hbox[4] = {64, static_cast<cuuint32_t>(p->halo_q),
                                static_cast<cuuint32_t>(p->halo_rows), 1};
    const cuuint32_t hes[4] = {1, 1, 1, 1};
    CUresult cr = encode(&ma.map,
                         is_int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         4, const_cast<void *>(act), hdim, hstride, hbox, hes,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         is_int8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS)
      return fail(FCONV_ERR_INTERNAL, "window tensor map encode failed (%d)", (int)cr);
    ma.base = act;
    ma.n = p->N;
    ma.form = a_form;
    ma.valid = true;
  }
  if (gather == fconv::Gather::kTmaIm2col &&
      !(ma.valid && ma.base == act && ma.n == p->N && ma.form == a_form)) {
    ma.valid = false;
    memset(&ma.map, 0, sizeof ma.map);
    CUtensorMap &tmap_a = ma.map;
    PFN_cuTensorMapEncodeIm2col_v12000 enc_a = encode_im2col_fn();
    if (!enc_a) return fail(FCONV_ERR_CUDA, "cuTensorMapEncodeIm2col is unavailable");
    // NHWC, innermost first: C, W, H, N.  The bounding box of filter-window
    // origins runs from -pad_before to (extent - 1) + pad_after - (filter - 1).
    const cuuint64_t adim[4] = {static_cast<cuuint64_t>(p->C), static_cast<cuuint64_t>(gW),
                                static_cast<cuuint64_t>(gH), static_cast<cuuint64_t>(p->N)};
    const cuuint64_t astride[3] = {static_cast<cuuint64_t>(p->C) * 2,
                                   static_cast<cuuint64_t>(gW) * p->C * 2,
                                   static_cast<cuuint64_t>(gH) * gW * p->C * 2};
    const int lower[2] = {-p->pl, -p->pt};
    const int upper[2] = {p->pr - (p->S - 1), p->pb - (p->R - 1)};
    const cuuint32_t traverse[4] = {1, static_cast<cuuint32_t>(gsw), static_cast<cuuint32_t>(gsh),
                                    1};
    // widening in the kernel: the int8 input itself, 64 one-byte channels a
    // pixel row, unswizzled (the converter warps lay it out for the MMA)
    const int elt = p->widen ? 1 : 2;
    const cuuint64_t astride_e[3] = {astride[0] / 2 * elt, astride[1] / 2 * elt,
                                     astride[2] / 2 * elt};
    CUresult cra = enc_a(&tmap_a,
                         p->widen ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : is_int8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         4, const_cast<void *>(act), adim, astride_e, lower, upper, 64,
                         static_cast<cuuint32_t>(a_pixels),
                         traverse, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         p->widen ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cra != CUDA_SUCCESS)
      return fail(FCONV_ERR_INTERNAL, "im2col tensor map encode failed (%d)", (int)cra);
    ma.base = act;
    ma.n = p->N;
    ma.form = a_form;
    ma.valid = true;
  }
  static const CUtensorMap kNoMap = {};
  const CUtensorMap &tmap_a =
      (gather == fconv::Gather::kTmaIm2col || halo) ? ma.map : kNoMap;

  fconv::ConvArgs a;
  memset(&a, 0, sizeof a);
  a.a = act;
  a.use_side = (mode == fconv::kModeFused && side != nullptr && side_scale != 0.0f) ? 1 : 0;
  a.side = a.use_side ? side : nullptr;
  a.bias = bias;
  a.scale_k = mode == fconv::kModeFused ? scale_k : nullptr;
  a.y = y;
  a.N = p->N; a.H = gH; a.W = gW; a.C = p->C; a.K = p->K; a.R = p->R; a.S = p->S;
  a.sh = gsh; a.sw = gsw; a.pt = p->pt; a.pl = p->pl; a.P = p->P; a.Q = p->Q;
  a.M = p->M;
  a.Ktot = p->Ktot;
  a.num_kb = p->num_kb;
  a.kb_chunk = p->kb_chunk;
  a.num_n_tiles = p->num_n_tiles;
  a.num_tiles = p->num_tiles;
  a.b3d = b3d;
  a.kps = kps;
  a.kdual = split_mma_issue(*p) ? 1 : 0;
  a.conv_scale = conv_scale;
  a.side_scale = side_scale;
  a.act = static_cast<int>(p->act);
  a.omap = p->omap; a.out_H = p->out_H; a.out_W = p->out_W;
  a.o_sh = p->o_sh; a.o_sw = p->o_sw; a.o_h0 = p->o_h0; a.o_w0 = p->o_w0;
  {
    const float inf = std::numeric_limits<float>::infinity();
    a.slope = 1.0f; a.lo = -inf; a.hi = inf;
    switch (p->act) {
      case FCONV_ACT_RELU: a.lo = 0.0f; break;
      case FCONV_ACT_LEAKY_RELU: a.slope = p->act_alpha; break;
      case FCONV_ACT_CLIPPED_RELU: a.lo = 0.0f; a.hi = p->act_alpha; break;
      case FCONV_ACT_CLAMP: a.lo = p->act_alpha; a.hi = p->act_beta; break;
      default: break;
    }
  }
  a.mode = mode;
  a.debug = p->debug;
  a.timeout_ns = static_cast<unsigned long long>(p->timeout_ms) * 1000000ull;
  a.splits = p->splits;
  a.kb_per_split = (p->num_kb + p->splits - 1) / p->splits;
  a.partial = split_partial;
  a.counters = split_counters;
  a.halo_q = p->halo_q;
  a.halo_tr = p->halo_tr;
  a.halo_rows = p->halo_rows;
  a.tiles_per_img = p->tiles_per_img;
  a.halo_slot = p->halo_slot;
  a.halo_stg = p->halo_stg;
  a.w_i8 = (halo && is_int8) ? static_cast<const int8_t *>(w) : nullptr;
  const long long units = static_cast<long long>(a.num_tiles) * a.splits;
  int grid = units < sms ? static_cast<int>(units) : sms;
  // the halo gather keeps each CTA on one output-channel tile
  if (halo) grid = grid / p->num_n_tiles * p->num_n_tiles;
  if (grid <= 0)
    return fail(FCONV_ERR_NOT_SUPPORTED, "%d output-channel tiles on %d SMs", p->num_n_tiles, sms);
  e = fconv::launch_conv(p->block_n, p->m_sub, is_int8, gather, tmap_a, tmap, a, grid,
                        /*overlap=*/prep, stream, p->widen != 0);
  if (e != cudaSuccess)
    return fail(FCONV_ERR_CUDA, "convolution launch: %s (%s)", cudaGetErrorString(e),
                fconv::last_launch_note());
  if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "event record");
  return FCONV_OK;
}

}  // namespace

namespace {

// The same convolution on the first n images of the batch (all derived
// extents recomputed; tile choice and workspace layout kept).
fconv_plan batch_slice(const fconv_plan &p, int n) {
  fconv_plan q = p;
  q.N = n;
  q.M = static_cast<long long>(n) * p.P * p.Q;
  q.num_tiles = tile_count(q);
  q.use_events = false;
  return q;
}

void destroy_pipeline(fconv_plan *p) {
  if (p->pipe_dev < 0) return;
  cudaStreamDestroy(p->s_in);
  cudaStreamDestroy(p->s_out);
  cudaEventDestroy(p->ev_entry);
  cudaEventDestroy(p->ev_out);
  for (int i = 0; i < kMaxHostChunks; ++i) {
    cudaEventDestroy(p->ev_in[i]);
    cudaEventDestroy(p->ev_comp[i]);
  }
  p->pipe_dev = -1;
}

void destroy_fork(fconv_plan *p) {
  if (p->fork_dev < 0) return;
  for (int i = 0; i < p->num_fork; ++i) {
    cudaStreamDestroy(p->fork_s[i]);
    cudaEventDestroy(p->fork_done[i]);
  }
  cudaEventDestroy(p->fork_start);
  p->fork_dev = -1;
  p->num_fork = 0;
}

// Side streams and events for the phases of a strided transposed plan, on
// the current device.
fconv_status ensure_fork(fconv_plan *p) {
  if (p->num_phases <= 1) return FCONV_OK;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->fork_dev == dev) return FCONV_OK;
  destroy_fork(p);
  const int n = p->num_phases - 1 < 3 ? p->num_phases - 1 : 3;
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaEventCreateWithFlags(&p->fork_start, ef) == cudaSuccess;
  int made = 0;
  for (; ok && made < n; ++made)
    ok = cudaStreamCreateWithFlags(&p->fork_s[made], cudaStreamNonBlocking) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->fork_done[made], ef) == cudaSuccess;
  if (!ok) {
    e = cudaGetLastError();
    return cuda_fail(e, "creating the phase streams");
  }
  p->num_fork = n;
  p->fork_dev = dev;
  return FCONV_OK;
}

// Streams and events for the host-buffer pipeline, on the current device.
fconv_status ensure_pipeline(fconv_plan *p) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (p->pipe_dev == dev) return FCONV_OK;
  destroy_pipeline(p);
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&p->ev_entry, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&p->ev_out, ef) == cudaSuccess;
  for (int i = 0; ok && i < kMaxHostChunks; ++i)
    ok = cudaEventCreateWithFlags(&p->ev_in[i], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->ev_comp[i], ef) == cudaSuccess;
  if (!ok) {
    e = cudaGetLastError();
    return cuda_fail(e, "creating the copy streams");
  }
  p->pipe_dev = dev;
  return FCONV_OK;
}

}  // namespace

namespace fconv {
// Record the detail fconv_last_error() returns, for other translation units.
fconv_status record_error(fconv_status st, const char *msg) { return fail(st, "%s", msg); }

// The fused run with a caller-chosen workspace, for other translation units
// of this library (the no-allocation entry point).
fconv_status enqueue_fused(fconv_plan *p, const void *x, const void *w, const float *bias,
                           const void *side, float conv_scale, float side_scale, void *y,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream) {
  return enqueue(p, x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
                 stream, kModeFused);
}
}  // namespace fconv

namespace {
fconv_status finish_plan(fconv_plan &p, fconv_plan **plan);
}  // namespace

extern "C" {

fconv_status fconv_plan_create(fconv_plan **plan, int N, int H, int W, int C, int K, int R, int S,
                               int stride_h, int stride_w, fconv_padding padding,
                               fconv_dtype dtype, fconv_act act) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan output pointer is NULL");
  *plan = nullptr;
  if (N <= 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0)
    return fail(FCONV_ERR_INVALID_VALUE, "every extent must be positive");
  if (stride_h <= 0 || stride_w <= 0) return fail(FCONV_ERR_INVALID_VALUE, "strides must be >= 1");
  if (padding != FCONV_SAME && padding != FCONV_VALID)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown padding %d", (int)padding);
  if (dtype != FCONV_INT8 && dtype != FCONV_BF16)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown dtype %d", (int)dtype);
  if (act < FCONV_ACT_NONE || act > FCONV_ACT_CLAMP)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown activation %d", (int)act);

  fconv_plan p;
  memset(&p, 0, sizeof p);
  p.N = N; p.H = H; p.W = W; p.C = C; p.K = K; p.R = R; p.S = S;
  p.sh = stride_h; p.sw = stride_w;
  p.padding = padding; p.dtype = dtype; p.act = act;
  if (!axis_geometry(H, R, stride_h, padding, &p.P, &p.pt, &p.pb) ||
      !axis_geometry(W, S, stride_w, padding, &p.Q, &p.pl, &p.pr))
    return fail(FCONV_ERR_INVALID_VALUE, "VALID padding with a filter larger than the input");

  return finish_plan(p, plan);
}

}  // extern "C"

namespace {

// Everything after the geometry: limits, k-blocks, tile, workspace.
fconv_status finish_plan(fconv_plan &p, fconv_plan **plan) {
  const int N = p.N, H = p.H, W = p.W, C = p.C, K = p.K, R = p.R, S = p.S;
  const fconv_dtype dtype = p.dtype;
  const int stride_h = p.sh, stride_w = p.sw;
  const int vec = dtype == FCONV_INT8 ? 16 : 8;
  if (C % vec != 0 || K % vec != 0)
    return fail(FCONV_ERR_NOT_SUPPORTED,
                "C and K must be multiples of %d for this dtype (16-byte vectors); got C=%d K=%d",
                vec, C, K);
  const long long in_elems = static_cast<long long>(N) * H * W * C;
  const long long out_elems = static_cast<long long>(N) * p.P * p.Q * K;
  const long long ktot = static_cast<long long>(R) * S * C;
  if (in_elems > kLimit || out_elems > kLimit || ktot * K > kLimit)
    return fail(FCONV_ERR_NOT_SUPPORTED, "a tensor has 2^31 or more elements");

  p.M = static_cast<long long>(N) * p.P * p.Q;
  p.Ktot = static_cast<int>(ktot);
  p.num_kb = (p.Ktot + 63) / 64;
  if (dtype == FCONV_INT8 && p.num_kb > fconv::kMaxExactKBlocks) {
    const int chunks = (p.num_kb + fconv::kMaxExactKBlocks - 1) / fconv::kMaxExactKBlocks;
    p.kb_chunk = (p.num_kb + chunks - 1) / chunks;
  } else {
    p.kb_chunk = p.num_kb;
  }
  const long long m_tiles = (p.M + 127) / 128;
  if (m_tiles * ((K + 31) / 32) > kLimit)
    return fail(FCONV_ERR_NOT_SUPPORTED, "too many output tiles");
  p.subsample =
      (!p.transposed && dtype == FCONV_INT8 && R == 1 && S == 1 && (stride_h > 1 || stride_w > 1))
          ? 1 : 0;
  // the phases of a strided transposed plan run concurrently (up to four
  // streams), each on its share of the SMs
  p.pack_filter = (dtype == FCONV_INT8 || p.tap_nR > 0) ? 1 : 0;
  const int sms = sm_count_of_current_device(148);
  const TileChoice tile = choose_tile(p, p.sm_share > 1 ? sms / p.sm_share : sms);
  p.auto_block_n = tile.bn;
  p.auto_m_sub = tile.ms;
  p.auto_splits = tile.splits;
  p.auto_halo = tile.halo;
  set_tiling(p, tile.bn, tile.ms, tile.splits, tile.halo);
  p.timeout_ms = 2000;
  p.host_chunks = 0;
  p.pipe_dev = -1;
  p.fork_dev = -1;
  p.wt_bytes = p.pack_filter ? align_up(static_cast<size_t>(K) * p.Ktot * 2, 256) : 0;
  const InputView view = input_view(p);
  const long long xh_elems = static_cast<long long>(N) * view.H * view.W * C;
  if (xh_elems > kLimit) return fail(FCONV_ERR_NOT_SUPPORTED, "a tensor has 2^31 or more elements");
  update_widen(p);
  p.ws_wt_off = 0;
  p.ws_xh_off = p.wt_bytes;

  fconv_plan *out = new (std::nothrow) fconv_plan(p);
  if (!out) return fail(FCONV_ERR_INTERNAL, "out of host memory");
  *plan = out;
  return FCONV_OK;
}

}  // namespace

extern "C" {

fconv_status fconv_plan_create_transposed(fconv_plan **plan, int N, int H, int W, int C, int K,
                                          int R, int S, int stride_h, int stride_w, int pad_top,
                                          int pad_bottom, int pad_left, int pad_right,
                                          fconv_dtype dtype, fconv_act act) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan output pointer is NULL");
  *plan = nullptr;
  if (N <= 0 || H <= 0 || W <= 0 || C <= 0 || K <= 0 || R <= 0 || S <= 0)
    return fail(FCONV_ERR_INVALID_VALUE, "every extent must be positive");
  if (stride_h <= 0 || stride_w <= 0) return fail(FCONV_ERR_INVALID_VALUE, "strides must be >= 1");
  if (dtype != FCONV_INT8 && dtype != FCONV_BF16)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown dtype %d", (int)dtype);
  if (act < FCONV_ACT_NONE || act > FCONV_ACT_CLAMP)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown activation %d", (int)act);
  const long long Ho = static_cast<long long>(H - 1) * stride_h + R - pad_top - pad_bottom;
  const long long Wo = static_cast<long long>(W - 1) * stride_w + S - pad_left - pad_right;
  if (Ho <= 0 || Wo <= 0) return fail(FCONV_ERR_INVALID_VALUE, "the pads leave no output");
  // pads in [0, filter-1]; the bottom/right pad may go down to 1-stride
  // (an output adjustment larger than the pad)
  if (pad_top < 0 || pad_top > R - 1 || pad_bottom < 1 - stride_h || pad_bottom > R - 1 ||
      pad_left < 0 || pad_left > S - 1 || pad_right < 1 - stride_w || pad_right > S - 1)
    return fail(FCONV_ERR_NOT_SUPPORTED,
                "transposed-convolution pads must lie in [0, filter-1] (bottom/right down to "
                "1-stride)");
  if (stride_h > 8 || stride_w > 8)
    return fail(FCONV_ERR_NOT_SUPPORTED, "transposed-convolution strides above 8");
  // Stride 1: out[h, w] = sum over taps of x[h - r + pad_top, w - s + pad_left] w[r, s]
  // is the cross-correlation of x with the filter flipped in both spatial
  // axes and padded by filter-1-pad on each side.  Stride s <= filter: the
  // output splits into s*s phases (rows ho with (ho + pad_top) % sh = a,
  // columns likewise with b); phase (a, b) gets only the taps r = a + sh*j,
  // s = b + sw*l, and is the stride-1 cross-correlation of x with those taps
  // flipped, writing every sh-th row and sw-th column.  Stride > filter: the
  // stride-1 case on x with zero rows/columns inserted (some outputs get no
  // tap at all there).
  fconv_plan p;
  memset(&p, 0, sizeof p);
  p.N = N; p.H = H; p.W = W; p.C = C; p.K = K; p.R = R; p.S = S;
  p.sh = stride_h; p.sw = stride_w;
  const bool strided = stride_h > 1 || stride_w > 1;
  const bool phased = strided && R >= stride_h && S >= stride_w;
  p.upsample = (strided && !phased) ? 1 : 0;
  p.padding = FCONV_VALID;   // unused: the pads are explicit
  p.dtype = dtype; p.act = act;
  p.transposed = 1;
  p.tpad[0] = pad_top; p.tpad[1] = pad_bottom; p.tpad[2] = pad_left; p.tpad[3] = pad_right;
  p.pt = R - 1 - pad_top; p.pb = R - 1 - pad_bottom;
  p.pl = S - 1 - pad_left; p.pr = S - 1 - pad_right;
  p.P = static_cast<int>(Ho);
  p.Q = static_cast<int>(Wo);
  p.tap_nR = R; p.tap_nS = S; p.tap_R = R; p.tap_S = S;   // flipped filter
  p.tap_rstep = 1; p.tap_sstep = 1;
  if (!phased) return finish_plan(p, plan);

  // the phases: forward plans over x (stride 1, explicit pads)
  auto floor_div = [](long long a, long long b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
  auto ceil_div = [&](long long a, long long b) { return -floor_div(-a, b); };
  fconv_plan *phases[64];
  int np = 0;
  auto cleanup = [&]() {
    for (int i = 0; i < np; ++i) delete phases[i];
  };
  size_t wt_total = 0;
  for (int a = 0; a < stride_h; ++a) {
    for (int b = 0; b < stride_w; ++b) {
      const int Ra = (R - a + stride_h - 1) / stride_h, Sb = (S - b + stride_w - 1) / stride_w;
      const long long u_lo = ceil_div(pad_top - a, stride_h);
      const long long u_hi = floor_div(Ho - 1 + pad_top - a, stride_h);
      const long long v_lo = ceil_div(pad_left - b, stride_w);
      const long long v_hi = floor_div(Wo - 1 + pad_left - b, stride_w);
      if (u_hi < u_lo || v_hi < v_lo) continue;   // no output row or column in this phase
      fconv_plan q;
      memset(&q, 0, sizeof q);
      q.N = N; q.H = H; q.W = W; q.C = C; q.K = K; q.R = Ra; q.S = Sb;
      q.sh = 1; q.sw = 1;
      q.padding = FCONV_VALID; q.dtype = dtype; q.act = act; q.transposed = 1;
      q.P = static_cast<int>(u_hi - u_lo + 1);
      q.Q = static_cast<int>(v_hi - v_lo + 1);
      // output p of the phase reads input rows p + j - pt, j < Ra
      q.pt = static_cast<int>(Ra - 1 - u_lo);
      q.pl = static_cast<int>(Sb - 1 - v_lo);
      q.pb = q.P - H - q.pt + Ra - 1;
      q.pr = q.Q - W - q.pl + Sb - 1;
      q.tap_nR = Ra; q.tap_nS = Sb; q.tap_R = R; q.tap_S = S;
      q.tap_r0 = a; q.tap_s0 = b; q.tap_rstep = stride_h; q.tap_sstep = stride_w;
      q.omap = 1; q.out_H = static_cast<int>(Ho); q.out_W = static_cast<int>(Wo);
      q.o_sh = stride_h; q.o_sw = stride_w;
      q.sm_share = stride_h * stride_w < 4 ? stride_h * stride_w : 4;
      q.o_h0 = static_cast<int>(stride_h * u_lo + a - pad_top);
      q.o_w0 = static_cast<int>(stride_w * v_lo + b - pad_left);
      fconv_plan *made = nullptr;
      const fconv_status st = finish_plan(q, &made);
      if (st != FCONV_OK) {
        cleanup();
        return st;
      }
      made->ws_wt_off = wt_total;
      wt_total += made->wt_bytes;
      phases[np++] = made;
    }
  }
  // the whole plan: the geometry above for checks and reports; its
  // workspace is the phases' filter copies, then one input copy (int8)
  fconv_plan *whole = nullptr;
  const fconv_status st = finish_plan(p, &whole);
  if (st != FCONV_OK) {
    cleanup();
    return st;
  }
  whole->num_phases = np;
  for (int i = 0; i < np; ++i) {
    whole->phase[i] = phases[i];
    phases[i]->ws_xh_off = wt_total;
  }
  whole->wt_bytes = wt_total;
  whole->ws_wt_off = 0;
  whole->ws_xh_off = wt_total;
  whole->xh_bytes = dtype == FCONV_INT8 ? align_up(static_cast<size_t>(N) * H * W * C * 2, 256) : 0;
  for (int i = 0; i < np; ++i) phases[i]->xh_bytes = whole->xh_bytes;
  whole->num_tiles = 0;
  for (int i = 0; i < np; ++i) whole->num_tiles += phases[i]->num_tiles;
  whole->block_n = phases[0]->block_n;
  whole->kb_chunk = phases[0]->kb_chunk;
  *plan = whole;
  return FCONV_OK;
}

fconv_status fconv_plan_set_activation_params(fconv_plan *plan, float alpha, float beta) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (!std::isfinite(alpha) || !std::isfinite(beta))
    return fail(FCONV_ERR_INVALID_VALUE, "activation parameters must be finite");
  if (plan->act == FCONV_ACT_CLIPPED_RELU && alpha < 0.0f)
    return fail(FCONV_ERR_INVALID_VALUE, "clipped Relu needs alpha >= 0, got %g", alpha);
  if (plan->act == FCONV_ACT_CLAMP && alpha > beta)
    return fail(FCONV_ERR_INVALID_VALUE, "clamp needs alpha <= beta, got [%g, %g]", alpha, beta);
  plan->act_alpha = alpha;
  plan->act_beta = beta;
  return FCONV_OK;
}

fconv_status fconv_plan_destroy(fconv_plan *plan) {
  if (plan) {
    destroy_pipeline(plan);
    destroy_fork(plan);
    for (int i = 0; i < plan->num_phases; ++i) delete plan->phase[i];
  }
  delete plan;
  return FCONV_OK;
}

fconv_status fconv_fold_batchnorm(int K, float conv_scale, const float *bias, const float *gamma,
                                  const float *beta, const float *mean, const float *var,
                                  float eps, float *scale_out, float *bias_out) {
  if (K <= 0) return fail(FCONV_ERR_INVALID_VALUE, "K must be positive");
  if (!gamma || !beta || !mean || !var || !scale_out || !bias_out)
    return fail(FCONV_ERR_INVALID_VALUE, "gamma, beta, mean, var and the outputs must not be NULL");
  if (!std::isfinite(eps) || eps < 0.0f) return fail(FCONV_ERR_INVALID_VALUE, "eps must be >= 0");
  for (int k = 0; k < K; ++k)
    if (!(static_cast<double>(var[k]) + eps > 0.0))
      return fail(FCONV_ERR_INVALID_VALUE, "var + eps must be positive");
  for (int k = 0; k < K; ++k) {
    const double g = static_cast<double>(gamma[k]) / std::sqrt(static_cast<double>(var[k]) + eps);
    const double b = bias ? static_cast<double>(bias[k]) : 0.0;
    scale_out[k] = static_cast<float>(static_cast<double>(conv_scale) * g);
    bias_out[k] = static_cast<float>((b - static_cast<double>(mean[k])) * g + beta[k]);
  }
  return FCONV_OK;
}

fconv_status fconv_plan_output_shape(const fconv_plan *plan, int *N, int *P, int *Q, int *K) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (N) *N = plan->N;
  if (P) *P = plan->P;
  if (Q) *Q = plan->Q;
  if (K) *K = plan->K;
  return FCONV_OK;
}

fconv_status fconv_plan_padding(const fconv_plan *plan, int *pad_top, int *pad_bottom,
                                int *pad_left, int *pad_right) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  const bool t = plan->transposed != 0;   // report the pads the caller gave
  if (pad_top) *pad_top = t ? plan->tpad[0] : plan->pt;
  if (pad_bottom) *pad_bottom = t ? plan->tpad[1] : plan->pb;
  if (pad_left) *pad_left = t ? plan->tpad[2] : plan->pl;
  if (pad_right) *pad_right = t ? plan->tpad[3] : plan->pr;
  return FCONV_OK;
}

fconv_status fconv_workspace_size(const fconv_plan *plan, size_t *bytes) {
  if (!plan || !bytes) return fail(FCONV_ERR_INVALID_VALUE, "plan and bytes must not be NULL");
  *bytes = workspace_need(*plan);
  return FCONV_OK;
}

fconv_status fconv_run(fconv_plan *plan, const void *x, const void *w, const float *bias,
                       const void *side, float conv_scale, float side_scale, void *y,
                       void *workspace, size_t workspace_bytes, fconv_stream_t stream) {
  return enqueue(plan, x, w, bias, side, conv_scale, side_scale, y, workspace, workspace_bytes,
                 reinterpret_cast<cudaStream_t>(stream), fconv::kModeFused);
}

fconv_status fconv_run_channel_scale(fconv_plan *plan, const void *x, const void *w,
                                     const float *bias, const void *side,
                                     const float *conv_scale, float side_scale, void *y,
                                     void *workspace, size_t workspace_bytes,
                                     fconv_stream_t stream) {
  if (!conv_scale) return fail(FCONV_ERR_INVALID_VALUE, "conv_scale must not be NULL");
  return enqueue(plan, x, w, bias, side, 0.0f, side_scale, y, workspace, workspace_bytes,
                 reinterpret_cast<cudaStream_t>(stream), fconv::kModeFused, false, conv_scale);
}

fconv_status fconv_run_accumulators(fconv_plan *plan, const void *x, const void *w, void *acc,
                                    void *workspace, size_t workspace_bytes,
                                    fconv_stream_t stream) {
  return enqueue(plan, x, w, nullptr, nullptr, 1.0f, 0.0f, acc, workspace, workspace_bytes,
                 reinterpret_cast<cudaStream_t>(stream), fconv::kModeAccumulators);
}

static void host_layout(const fconv_plan *p, int with_side, size_t off[6]) {
  const size_t elt = p->dtype == FCONV_INT8 ? 1 : 2;
  const size_t x_b = static_cast<size_t>(p->N) * p->H * p->W * p->C * elt;
  const size_t w_b = static_cast<size_t>(p->R) * p->S * p->C * p->K * elt;
  const size_t b_b = static_cast<size_t>(p->K) * 4;
  const size_t y_b = static_cast<size_t>(p->M) * p->K * elt;
  off[0] = 0;                                                 // workspace
  off[1] = align_up(off[0] + workspace_need(*p), 256);         // x
  off[2] = align_up(off[1] + x_b, 256);                        // w
  off[3] = align_up(off[2] + w_b, 256);                        // bias
  off[4] = align_up(off[3] + b_b, 256);                        // side
  off[5] = align_up(off[4] + (with_side ? y_b : 0), 256);      // y
  (void)y_b;
}

fconv_status fconv_host_workspace_size(const fconv_plan *plan, int with_side, size_t *bytes) {
  if (!plan || !bytes) return fail(FCONV_ERR_INVALID_VALUE, "plan and bytes must not be NULL");
  size_t off[6];
  host_layout(plan, with_side, off);
  const size_t elt = plan->dtype == FCONV_INT8 ? 1 : 2;
  *bytes = align_up(off[5] + static_cast<size_t>(plan->M) * plan->K * elt, 256);
  return FCONV_OK;
}

// Image counts of the batch chunks fconv_run_host pipelines over, in order
// (they sum to N); returns how many.  Copy-in of chunk i+1 and copy-out of
// chunk i-1 overlap the compute of chunk i, and the host link bounds the
// whole run, so what is not hidden is the copy-in of the first chunk and
// the compute and copy-out of the last.  A fixed count (host_chunks > 0)
// splits the batch evenly.  Automatic, with W(k) the most images whose
// output tiles fill at most k waves (one tile per SM): a batch of at least
// ten W(1) ramps up through W(1)/6, W(1)/2 and W(2) images, runs middle
// chunks of at most W(3), and ramps down through W(2), W(1) and 2 W(1)/3.
// The first compute then starts after a short copy, each chunk of the
// ramp-down computes in about the time the next one takes to copy in, and
// the last chunk's compute and copy-out are short; a chunk one image past
// a whole number of waves costs a wave more.  (N=256 28x28x512 int8 on 152
// SMs: 2, 6, 24, 36 x 5, 24, 12, 8 ran 1.26 ms against 1.30-1.31 for
// twelve even chunks and 1.28 for the same ramp with chunks of 25 and 35.)
// A smaller batch takes even chunks of at least one wave each, up to 12
// (4 chunks 1.44 ms, 8 1.34, 12 1.33, 16 1.36 on the same layer), and one
// chunk when it has less.
int host_chunk_sizes(const fconv_plan &p, int sms, int sizes[kMaxHostChunks]) {
  const int N = p.N;
  auto even = [&](int chunks) {
    chunks = std::max(1, std::min({chunks, kMaxHostChunks, N}));
    const int per = (N + chunks - 1) / chunks;
    int count = 0;
    for (int left = N; left > 0; left -= per) sizes[count++] = std::min(per, left);
    return count;
  };
  if (p.host_chunks > 0) return even(p.host_chunks);
  if (sms <= 0 || p.num_tiles <= 0) return even(1);
  // output tiles of an n-image slice (a plan of sub-pixel phases: in proportion)
  auto tiles = [&](int n) -> long long {
    if (p.num_phases > 0)
      return (static_cast<long long>(p.num_tiles) * n + N - 1) / N;
    return batch_slice(p, n).num_tiles;
  };
  auto most_images = [&](int waves) {   // W(waves), 0 if one image needs more
    const long long cap = static_cast<long long>(waves) * sms;
    int lo = 0, hi = N;
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (tiles(mid) <= cap) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  const int w1 = most_images(1);
  if (w1 < 1 || N < 10 * w1) return even(std::min(12, p.num_tiles / sms));
  const int w2 = most_images(2), w3 = most_images(3);
  const int head[3] = {std::max(1, w1 / 6), std::max(1, w1 / 2), w2};
  const int tail[3] = {w2, w1, std::max(1, 2 * w1 / 3)};
  int fixed = 0;
  for (int v : head) fixed += v;
  for (int v : tail) fixed += v;
  const int rest = N - fixed;   // about 10 W(1) - 6.3 W(1)
  if (rest < 1) return even(std::min(12, p.num_tiles / sms));
  const int mids = std::min(kMaxHostChunks - 6, (rest + w3 - 1) / w3);
  int count = 0;
  for (int v : head) sizes[count++] = v;
  for (int i = 0; i < mids; ++i) sizes[count++] = rest / mids + (i < rest % mids ? 1 : 0);
  for (int v : tail) sizes[count++] = v;
  return count;
}

fconv_status fconv_plan_host_chunk_sizes(const fconv_plan *plan, int sm_count, int *sizes,
                                         int max_sizes, int *count) {
  if (!plan || !count) return fail(FCONV_ERR_INVALID_VALUE, "plan and count must not be NULL");
  if (sm_count <= 0) return fail(FCONV_ERR_INVALID_VALUE, "sm_count must be positive");
  int tmp[kMaxHostChunks];
  const int n = host_chunk_sizes(*plan, sm_count, tmp);
  *count = n;
  if (sizes) {
    if (max_sizes < n) return fail(FCONV_ERR_INVALID_VALUE, "%d chunks need %d entries", n, n);
    for (int i = 0; i < n; ++i) sizes[i] = tmp[i];
  }
  return FCONV_OK;
}

fconv_status fconv_run_host(fconv_plan *plan, const void *x_host, const void *w_host,
                            const float *bias_host, const void *side_host, float conv_scale,
                            float side_scale, void *y_host, void *device_workspace,
                            size_t workspace_bytes, fconv_stream_t stream) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (!x_host || !w_host || !bias_host || !y_host)
    return fail(FCONV_ERR_INVALID_VALUE, "x, w, bias and y must not be NULL");
  size_t need = 0;
  fconv_host_workspace_size(plan, side_host != nullptr, &need);
  if (!device_workspace || workspace_bytes < need)
    return fail(FCONV_ERR_WORKSPACE, "device workspace of %zu bytes needed", need);
  if (!aligned(device_workspace, 256))
    return fail(FCONV_ERR_MISALIGNED, "device workspace must be 256-byte aligned");
  size_t off[6];
  host_layout(plan, side_host != nullptr, off);
  uint8_t *base = static_cast<uint8_t *>(device_workspace);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t elt = plan->dtype == FCONV_INT8 ? 1 : 2;
  const size_t img_x = static_cast<size_t>(plan->H) * plan->W * plan->C * elt;
  const size_t img_y = static_cast<size_t>(plan->P) * plan->Q * plan->K * elt;
  const size_t w_b = static_cast<size_t>(plan->R) * plan->S * plan->C * plan->K * elt;

  int sizes[kMaxHostChunks];
  const int chunks = host_chunk_sizes(*plan, device_sm_count(nullptr), sizes);

  fconv_status s = ensure_pipeline(plan);
  if (s != FCONV_OK) return s;
  // the phase streams of a strided transposed plan belong to the plan, not
  // to the per-chunk copies below
  if ((s = ensure_fork(plan)) != FCONV_OK) return s;
  cudaError_t e;
  // the copy streams start after everything already queued on the caller's stream
  if ((e = cudaEventRecord(plan->ev_entry, st)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(plan->s_in, plan->ev_entry, 0)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(plan->s_out, plan->ev_entry, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  if ((e = cudaMemcpyAsync(base + off[2], w_host, w_b, cudaMemcpyHostToDevice, plan->s_in)) !=
          cudaSuccess ||
      (e = cudaMemcpyAsync(base + off[3], bias_host, static_cast<size_t>(plan->K) * 4,
                           cudaMemcpyHostToDevice, plan->s_in)) != cudaSuccess)
    return cuda_fail(e, "host-to-device copy");
  for (int i = 0, first = 0; i < chunks; first += sizes[i++]) {
    const size_t n0 = static_cast<size_t>(first);
    const size_t n = static_cast<size_t>(sizes[i]);
    if ((e = cudaMemcpyAsync(base + off[1] + n0 * img_x, static_cast<const uint8_t *>(x_host) +
                                 n0 * img_x, n * img_x, cudaMemcpyHostToDevice, plan->s_in)) !=
        cudaSuccess)
      return cuda_fail(e, "host-to-device copy");
    if (side_host &&
        (e = cudaMemcpyAsync(base + off[4] + n0 * img_y, static_cast<const uint8_t *>(side_host) +
                                 n0 * img_y, n * img_y, cudaMemcpyHostToDevice, plan->s_in)) !=
            cudaSuccess)
      return cuda_fail(e, "host-to-device copy of the side input");
    if ((e = cudaEventRecord(plan->ev_in[i], plan->s_in)) != cudaSuccess)
      return cuda_fail(e, "event record");
  }
  for (int i = 0, first = 0; i < chunks; first += sizes[i++]) {
    const size_t n0 = static_cast<size_t>(first);
    const int n = sizes[i];
    if ((e = cudaStreamWaitEvent(st, plan->ev_in[i], 0)) != cudaSuccess)
      return cuda_fail(e, "stream ordering");
    fconv_plan q = batch_slice(*plan, n);
    s = enqueue(&q, base + off[1] + n0 * img_x, base + off[2],
                reinterpret_cast<const float *>(base + off[3]),
                side_host ? base + off[4] + n0 * img_y : nullptr, conv_scale, side_scale,
                base + off[5] + n0 * img_y, base, off[1], st, fconv::kModeFused,
                /*skip_pack=*/i > 0);
    if (s != FCONV_OK) return s;
    if ((e = cudaEventRecord(plan->ev_comp[i], st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(plan->s_out, plan->ev_comp[i], 0)) != cudaSuccess)
      return cuda_fail(e, "stream ordering");
    if ((e = cudaMemcpyAsync(static_cast<uint8_t *>(y_host) + n0 * img_y,
                             base + off[5] + n0 * img_y, n * img_y, cudaMemcpyDeviceToHost,
                             plan->s_out)) != cudaSuccess)
      return cuda_fail(e, "device-to-host copy");
  }
  // the caller's stream continues once the last result byte is on the host
  if ((e = cudaEventRecord(plan->ev_out, plan->s_out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(st, plan->ev_out, 0)) != cudaSuccess)
    return cuda_fail(e, "stream ordering");
  return FCONV_OK;
}

fconv_status fconv_plan_set_host_chunks(fconv_plan *plan, int chunks) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (chunks < 0 || chunks > kMaxHostChunks)
    return fail(FCONV_ERR_INVALID_VALUE, "chunks must be 0 (automatic) .. %d", kMaxHostChunks);
  plan->host_chunks = chunks;
  return FCONV_OK;
}

fconv_status fconv_plan_check(fconv_plan *plan, fconv_stream_t stream) {
  (void)plan;
  unsigned int st = 0;
  cudaError_t e = fconv::status_read_and_clear(reinterpret_cast<cudaStream_t>(stream), &st);
  if (e != cudaSuccess) return cuda_fail(e, "stream");
  if (st != 0)
    return fail(static_cast<fconv_status>(st), "a kernel reported %s",
                fconv_status_string(static_cast<fconv_status>(st)));
  return FCONV_OK;
}

fconv_status fconv_plan_set_tile(fconv_plan *plan, int block_n) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (plan->num_phases > 0) {
    // every phase takes the tile (or its own automatic choice for 0)
    for (int i = 0; i < plan->num_phases; ++i) {
      const fconv_status st = fconv_plan_set_tile(plan->phase[i], block_n);
      if (st != FCONV_OK) return st;
    }
    plan->block_n = plan->phase[0]->block_n;
    plan->num_tiles = 0;
    for (int i = 0; i < plan->num_phases; ++i) plan->num_tiles += plan->phase[i]->num_tiles;
    return FCONV_OK;
  }
  if (block_n == 0) {
    set_tiling(*plan, plan->auto_block_n, plan->auto_m_sub, plan->auto_splits,
               plan->gather_mode == FCONV_GATHER_IM2COL ? 0 : plan->auto_halo);
    return FCONV_OK;
  }
  if (block_n != 64 && block_n != 128 && block_n != 256)
    return fail(FCONV_ERR_NOT_SUPPORTED, "tile %d: this build has 64, 128 and 256", block_n);
  if (!fconv::gather_supports(gather_for(*plan, block_n, false), block_n,
                              plan->kb_chunk < plan->num_kb))
    return fail(FCONV_ERR_NOT_SUPPORTED,
                "tile %d leaves no tensor memory for the int32 sums this plan needs", block_n);
  set_tiling(*plan, block_n, 1, 1, 0);
  return FCONV_OK;
}

fconv_status fconv_plan_set_tile_shape(fconv_plan *plan, int pixels, int channels) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (pixels != 128 && pixels != 256)
    return fail(FCONV_ERR_NOT_SUPPORTED, "tiles of %d output pixels: 128 or 256", pixels);
  if (plan->num_phases > 0) {
    for (int i = 0; i < plan->num_phases; ++i) {
      const fconv_status st = fconv_plan_set_tile_shape(plan->phase[i], pixels, channels);
      if (st != FCONV_OK) return st;
    }
    plan->block_n = plan->phase[0]->block_n;
    plan->num_tiles = 0;
    for (int i = 0; i < plan->num_phases; ++i) plan->num_tiles += plan->phase[i]->num_tiles;
    return FCONV_OK;
  }
  const int ms = pixels / 128;
  if (plan->gather_mode == FCONV_GATHER_HALO && channels == 64 &&
      halo_geometry(*plan, ms, nullptr)) {
    set_tiling(*plan, 64, ms, 1, 1);   // the halo tile of that height
    return FCONV_OK;
  }
  if (!fconv::gather_supports(gather_for(*plan, channels, false), channels,
                              plan->kb_chunk < plan->num_kb, ms))
    return fail(FCONV_ERR_NOT_SUPPORTED, "no kernel for %d x %d tiles on this plan", pixels,
                channels);
  set_tiling(*plan, channels, ms, 1, 0);
  return FCONV_OK;
}

fconv_status fconv_plan_set_splits(fconv_plan *plan, int splits) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (splits < 0 || splits > kMaxSplits)
    return fail(FCONV_ERR_INVALID_VALUE, "splits %d: 0 (automatic) or 1 to %d", splits, kMaxSplits);
  if (splits == 0) {
    set_tiling(*plan, plan->auto_block_n, plan->auto_m_sub, plan->auto_splits,
               plan->gather_mode == FCONV_GATHER_IM2COL ? 0 : plan->auto_halo);
    return FCONV_OK;
  }
  if (splits > 1) {
    if (plan->transposed || plan->num_phases > 0)
      return fail(FCONV_ERR_NOT_SUPPORTED, "split-K is for forward convolution plans");
    if (gather_for(*plan, plan->block_n, false) != fconv::Gather::kTmaIm2col)
      return fail(FCONV_ERR_NOT_SUPPORTED, "split-K runs on the TMA im2col gather only");
    if (plan->m_sub != 1)
      return fail(FCONV_ERR_NOT_SUPPORTED, "split-K runs on 128-pixel tiles");
    if (splits > plan->num_kb)
      return fail(FCONV_ERR_NOT_SUPPORTED, "%d splits of %d k-blocks", splits, plan->num_kb);
  }
  set_tiling(*plan, plan->block_n, plan->m_sub, splits, splits == 1 ? plan->halo : 0);
  return FCONV_OK;
}

fconv_status fconv_plan_get_splits(const fconv_plan *plan, int *splits) {
  if (!plan || !splits) return fail(FCONV_ERR_INVALID_VALUE, "plan and splits must not be NULL");
  *splits = plan->splits > 0 ? plan->splits : 1;
  return FCONV_OK;
}

fconv_status fconv_plan_get_config(const fconv_plan *plan, int *block_n, int *kblocks_per_chunk,
                                   int *num_tiles) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (block_n) *block_n = plan->block_n;
  if (kblocks_per_chunk) *kblocks_per_chunk = plan->kb_chunk;
  if (num_tiles) *num_tiles = plan->num_tiles;
  return FCONV_OK;
}

fconv_status fconv_plan_set_timeout_ms(fconv_plan *plan, uint32_t ms) {
  if (!plan || ms == 0) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL or timeout is 0");
  plan->timeout_ms = ms;
  return FCONV_OK;
}

fconv_status fconv_plan_set_debug(fconv_plan *plan, int flags) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (flags & ~(FCONV_DEBUG_DROP_ARRIVE | FCONV_DEBUG_GATHER_CPASYNC |
                FCONV_DEBUG_ONE_KBLOCK_STAGES | FCONV_DEBUG_ONE_MMA_ISSUER))
    return fail(FCONV_ERR_INVALID_VALUE, "unknown flags");
  plan->debug = flags;
  if (plan->num_phases == 0) update_widen(*plan);
  return FCONV_OK;
}

fconv_status fconv_plan_set_input_widening(fconv_plan *plan, int mode) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (mode != FCONV_WIDEN_AUTO && mode != FCONV_WIDEN_IN_KERNEL && mode != FCONV_WIDEN_COPY)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown widening mode %d", mode);
  plan->widen_mode = mode;
  if (plan->num_phases == 0) {
    // the halo gather widens int8 windows in the kernel: the fp16 copy
    // moves the plan off it
    if (plan->halo && !halo_geometry(*plan, plan->m_sub, nullptr)) retile_without_halo(*plan);
    update_widen(*plan);
  }
  return FCONV_OK;
}

fconv_status fconv_plan_get_input_widening(const fconv_plan *plan, int *in_kernel) {
  if (!plan || !in_kernel)
    return fail(FCONV_ERR_INVALID_VALUE, "plan and in_kernel must not be NULL");
  // the halo gather widens int8 windows inside the kernel too
  *in_kernel = (plan->widen || (plan->dtype == FCONV_INT8 && halo_run(*plan))) ? 1 : 0;
  return FCONV_OK;
}

fconv_status fconv_plan_set_gather(fconv_plan *plan, int mode) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (mode != FCONV_GATHER_AUTO && mode != FCONV_GATHER_IM2COL && mode != FCONV_GATHER_HALO)
    return fail(FCONV_ERR_INVALID_VALUE, "unknown gather mode %d", mode);
  if (plan->num_phases > 0) {
    if (mode == FCONV_GATHER_HALO)
      return fail(FCONV_ERR_NOT_SUPPORTED, "the halo gather is for forward stride-1 plans");
    return FCONV_OK;
  }
  if (mode == FCONV_GATHER_HALO) {
    // the halo tile the automatic choice would take, else 256 pixels if
    // they fit, else 128
    int ms = plan->auto_halo ? plan->auto_m_sub : 2;
    if (!halo_geometry(*plan, ms, nullptr)) ms = 1;
    if (!halo_geometry(*plan, ms, nullptr))
      return fail(FCONV_ERR_NOT_SUPPORTED,
                  "the halo gather needs a forward stride-1 plan with C == 64 (or 32, int8), "
                  "at most 9 filter taps, one exact accumulation and windows that fit %d "
                  "bytes of shared memory beside the filter tile", fconv::kHaloRegion);
    plan->gather_mode = mode;
    set_tiling(*plan, 64, ms, 1, 1);
    return FCONV_OK;
  }
  plan->gather_mode = mode;
  if (mode == FCONV_GATHER_IM2COL) {
    if (plan->halo) retile_without_halo(*plan);
    return FCONV_OK;
  }
  set_tiling(*plan, plan->auto_block_n, plan->auto_m_sub, plan->auto_splits, plan->auto_halo);
  return FCONV_OK;
}

fconv_status fconv_plan_set_stage_events(fconv_plan *plan, void *const events[4]) {
  if (!plan) return fail(FCONV_ERR_INVALID_VALUE, "plan is NULL");
  if (!events) {
    plan->use_events = false;
    return FCONV_OK;
  }
  for (int i = 0; i < 4; ++i)
    if (!events[i]) return fail(FCONV_ERR_INVALID_VALUE, "event %d is NULL", i);
  for (int i = 0; i < 4; ++i) plan->events[i] = static_cast<cudaEvent_t>(events[i]);
  plan->use_events = true;
  return FCONV_OK;
}

fconv_status fconv_plan_launch_count(const fconv_plan *plan, int *launches) {
  if (!plan || !launches) return fail(FCONV_ERR_INVALID_VALUE, "plan and launches must not be NULL");
  // per forward plan: the prep launch (a filter copy, an input copy or
  // split-K counters to zero), a tail widening launch when a dense int8
  // input is not a multiple of 64 elements, and the convolution
  auto one = [](const fconv_plan &p) {
    const long long n = static_cast<long long>(p.N) * p.H * p.W * p.C;
    const bool tail = p.dtype == FCONV_INT8 && !p.widen && !halo_run(p) && !p.subsample &&
                      !p.upsample && n % 64 != 0;
    const bool prep = filter_copy_bytes(p) > 0 || (p.dtype == FCONV_INT8 && !halo_run(p)) ||
                      p.upsample || p.splits > 1;
    return (prep ? 1 : 0) + (tail ? 1 : 0) + 1;
  };
  int total = 0;
  if (plan->num_phases > 0) {
    for (int i = 0; i < plan->num_phases; ++i) {
      const fconv_plan &q = *plan->phase[i];
      total += i == 0 ? one(q) : 2;
    }
  } else {
    total = one(*plan);
  }
  *launches = total;
  return FCONV_OK;
}

const char *fconv_plan_kernel(const fconv_plan *plan) {
  if (!plan) return "";
  if (plan->num_phases > 0) plan = plan->phase[0];
  if (halo_run(*plan)) return plan->m_sub == 2 ? "tma-halo-m256" : "tma-halo";
  if (gather_for_run(*plan) == fconv::Gather::kTmaIm2col && plan->m_sub == 2)
    return "tma-im2col-m256";
  if (gather_for_run(*plan) == fconv::Gather::kTmaIm2col) {
    if (split_mma_issue(*plan))
      return kblocks_per_stage(*plan) == 2 ? "tma-im2col-kb2-dual" : "tma-im2col-dual";
    return kblocks_per_stage(*plan) == 2 ? "tma-im2col-kb2" : "tma-im2col";
  }
  return "cp-async";
}

const char *fconv_status_string(fconv_status s) {
  switch (s) {
    case FCONV_OK: return "FCONV_OK";
    case FCONV_ERR_INVALID_VALUE: return "FCONV_ERR_INVALID_VALUE";
    case FCONV_ERR_NOT_SUPPORTED: return "FCONV_ERR_NOT_SUPPORTED";
    case FCONV_ERR_MISALIGNED: return "FCONV_ERR_MISALIGNED";
    case FCONV_ERR_CUDA: return "FCONV_ERR_CUDA";
    case FCONV_ERR_TIMEOUT: return "FCONV_ERR_TIMEOUT";
    case FCONV_ERR_INTERNAL: return "FCONV_ERR_INTERNAL";
    case FCONV_ERR_WORKSPACE: return "FCONV_ERR_WORKSPACE";
  }
  return "FCONV_ERR_UNKNOWN";
}

const char *fconv_last_error(void) { return t_last_error.c_str(); }

}  // extern "C"
