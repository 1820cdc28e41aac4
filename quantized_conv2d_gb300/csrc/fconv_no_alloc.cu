// fconv_run_no_alloc: the fused convolution with its scratch memory taken
// from a fixed array that this library holds on every device, so the call
// itself allocates nothing.
//
// Who needs this: callers that must not allocate device memory while they
// run -- a plugin inside an engine that owns the whole device-memory
// budget, a latency-bound loop where a cudaMalloc/cudaFree (which can
// synchronize the device) is not acceptable, or code that may only use the
// memory it reserved at start-up.  They still pass their own inputs and
// output; only the scratch (the 16-bit filter copy, and for int8 plans the
// fp16 copy of the input) lives here.
//
// Limit: kNoAllocScratchBytes (32 MiB) per device, reserved when the
// library's module is loaded on that device and held until the process
// exits (or until cudaDeviceReset, after which the next call finds the
// array in the device's new context).  Plans whose fconv_workspace_size() exceeds it are rejected with
// FCONV_ERR_WORKSPACE.
//
// Sharing: every call on a device uses the same array, and the array keeps
// whatever the previous call left in it.  Nothing needs to start at zero:
// each call writes every scratch byte its kernels read (the prep launch
// writes every row of the filter copy, the whole input copy and the split-K
// counters; the convolution writes each partial sum before the last unit of
// its tile reads it) before reading it.  Calls whose
// kernels overlap on the GPU (different streams, or several host threads)
// race on the array; serialize them, e.g. on one stream.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "fconv.h"
#include "fconv_internal.h"

namespace fconv {
fconv_status record_error(fconv_status st, const char *msg);
fconv_status enqueue_fused(fconv_plan *p, const void *x, const void *w, const float *bias,
                           const void *side, float conv_scale, float side_scale, void *y,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);
}

namespace {

constexpr size_t kNoAllocScratchBytes = 32u << 20;

// The scratch itself: a file-scope device array.  In host code this name is
// only a stand-in for the symbol; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchEntry {
  void *addr;                  // device address of the array in that context
  unsigned long long ctx_id;   // the context it belongs to (0: not known)
};
ScratchEntry g_scratch[kMaxDevices] = {};

// The driver's unique id of the calling thread's current context, or 0 when
// there is none (or the driver cannot say).  cudaDeviceReset destroys a
// device's primary context; the next runtime call makes a new one, with a
// new id, in which the module (and this array) is loaded afresh, possibly
// at another address.
unsigned long long current_context_id() {
  static std::once_flag once;
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch on the current device, looked up once per
// device and context (with that device current) and cached.  If the
// context's id cannot be read, the address is looked up on every call.
fconv_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fconv::record_error(FCONV_ERR_CUDA, "no usable current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchEntry &e = g_scratch[dev];
  const unsigned long long ctx = current_context_id();
  if (!e.addr || ctx == 0 || e.ctx_id != ctx) {
    void *ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_no_alloc_scratch);
    if (err != cudaSuccess || !ptr) {
      cudaGetLastError();
      e.addr = nullptr;
      return fconv::record_error(FCONV_ERR_CUDA,
                                 "cudaGetSymbolAddress of the built-in scratch failed");
    }
    e.addr = ptr;
    // the lookup made the device's primary context current if none was
    e.ctx_id = ctx != 0 ? ctx : current_context_id();
  }
  *out = e.addr;
  return FCONV_OK;
}

}  // namespace

extern "C" fconv_status fconv_run_no_alloc(fconv_plan *plan, const void *x, const void *w,
                                           const float *bias, const void *side, float conv_scale,
                                           float side_scale, void *y, fconv_stream_t stream) {
  size_t need = 0;
  fconv_status s = fconv_workspace_size(plan, &need);
  if (s != FCONV_OK) return s;
  if (need > kNoAllocScratchBytes)
    return fconv::record_error(FCONV_ERR_WORKSPACE,
                               "this plan needs more scratch than the 32 MiB built-in array "
                               "(see fconv_workspace_size); use fconv_run with a workspace");
  void *scratch = nullptr;
  s = scratch_address(&scratch);
  if (s != FCONV_OK) return s;
  return fconv::enqueue_fused(plan, x, w, bias, side, conv_scale, side_scale, y, scratch,
                              kNoAllocScratchBytes, reinterpret_cast<cudaStream_t>(stream));
}
