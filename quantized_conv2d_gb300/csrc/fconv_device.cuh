// Device primitives for sm_103a: mbarriers with bounded waits, cp.async,
// TMA tiled loads, tcgen05 (TMEM allocation, MMA, commit, loads/stores) and
// the shared-memory matrix / instruction descriptors the MMA reads.
//
// Every wait here has a time limit.  A wait that runs out sets the CTA's
// abort flag and the device status word and returns false; later waits in
// the same CTA see the flag and return false at once, so every role leaves
// its loop, the CTA reaches its final barrier, frees its TMEM and exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace fconv {

// Device status word (one per device): 0 = fine, else an fconv_status code.
// The host reads and clears it in fconv_plan_check().  This header is
// included by exactly one translation unit, which owns the definition.
__device__ unsigned int g_status = 0;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// timeout_ns.  Returns false if the CTA is aborting or the limit ran out
// (then the abort flag and the device status word are set).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          volatile int *abort_flag,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort_flag) return false;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        atomicCAS(&g_status, 0u, 5u /* FCONV_ERR_TIMEOUT */);
        return false;
      }
    }
  }
}

// mbar_wait executed by every lane of a warp, which then takes lane 0's
// answer: the loop around it stays warp-uniform, so the descriptors and
// coordinates computed from its state stay warp-uniform too.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               volatile int *abort_flag,
                                               uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Two phases at once (the second only if `both`): in the steady state,
// where neither has to wait, the ready test of both barriers costs one
// round trip.
__device__ __forceinline__ bool mbar_wait2_warp(uint32_t bar0, uint32_t parity0, uint32_t bar1,
                                                uint32_t parity1, bool both,
                                                volatile int *abort_flag,
                                                uint64_t timeout_ns) {
  const bool r0 = mbar_try_wait(bar0, parity0);
  const bool r1 = !both || mbar_try_wait(bar1, parity1);
  if (__shfl_sync(0xffffffffu, (r0 && r1) ? 1 : 0, 0) != 0) return true;
  if (!mbar_wait_warp(bar0, parity0, abort_flag, timeout_ns)) return false;
  return !both || mbar_wait_warp(bar1, parity1, abort_flag, timeout_ns);
}

// A wait used only while shutting down after an abort: ignores the abort
// flag, gives up silently after timeout_ns.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity,
                                                uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// ---------------------------------------------------------------- cp.async
// 16-byte copy global -> shared; src_bytes 0 writes 16 zero bytes.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the
// async proxy (the tensor core reads operands through it).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- launch order
// Programmatic dependent launch: a convolution launch may begin (barrier
// set-up, tensor-memory allocation, descriptor prefetch) while the prep
// launch before it in the stream still runs.  griddep_wait blocks until that
// grid has completed and its writes are visible; threads that read what it
// wrote call it first.  griddep_launch_dependents lets the next launch start
// once every block of this grid has called it (or finished).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled load of the box at (c0 = innermost, c1) into shared memory,
// completing `bar`'s transaction count.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0,
                                            int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// 3-D tiled load of the box at (c0 = innermost, c1, c2).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// A 4-D tiled box (coordinates innermost first); parts of the box outside
// the tensor (negative or past the extent) read as zero.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}

// 4-D im2col load (NHWC tensor map): pixelsPerColumn output pixels starting
// at the filter-window origin (w, h, n) of the first one, walking the
// tensor map's bounding box with its traversal strides, each pixel shifted by
// the filter tap (off_w, off_h); channelsPerPixel channels from c.  Pixels
// outside the tensor read as zero.  c * element size must be a multiple of
// 16 bytes.
__device__ __forceinline__ void tma_load_im2col_4d(uint32_t dst, const CUtensorMap *map, int c,
                                                   int w, int h, int n, uint16_t off_w,
                                                   uint16_t off_h, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.im2col.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], {%7, %8};" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c), "r"(w), "r"(h), "r"(n), "r"(bar),
      "h"(off_w), "h"(off_h)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, 16-bit inputs, fp32 accumulate.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all tcgen05 operations this thread issued
// before have completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

#define FCONV_R32(v)                                                                      \
  "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),     \
      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),          \
      "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]),       \
      "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),       \
      "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]),       \
      "=r"(v[31])
#define FCONV_RW32(v)                                                                     \
  "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),     \
      "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]),          \
      "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]),       \
      "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]),       \
      "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]),       \
      "+r"(v[31])
#define FCONV_IN32(v)                                                                     \
  "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), \
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),   \
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),  \
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),  \
      "r"(v[29]), "r"(v[30]), "r"(v[31])

// Warp-collective: lane i reads TMEM lane (taddr.lane + i), 32 consecutive
// 32-bit columns starting at taddr.col.  The values are valid only after
// tmem_wait_ld(v), which also orders every later use of v after the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : FCONV_R32(v)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : FCONV_RW32(v)::"memory");
}

// Warp-collective store of 32 consecutive columns per lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      FCONV_IN32(v)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored with
// the 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart.
// The tile base must be 1024-byte aligned; stepping K by 16 elements
// (32 bytes) inside the atom adds 2 to the start-address field.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                      // leading offset (unused)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride offset: 8 rows
  d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
  return d;
}

// The same descriptor for a tile that starts `row` 128-byte rows into a
// 1024-byte-aligned buffer written with the 128-byte swizzle (a TMA copy
// XORs each row's 16-byte chunk index with bits 7-9 of the row's address).
// A start inside an 8-row atom needs nothing more: the MMA takes the XOR
// pattern from the same address bits of each row it reads, so the
// base-offset field stays 0.  (Measured on GB300: with that field set to
// the start's row within its atom, (address >> 7) & 7, every sum came out
// wrong; with 0 the sums of every tap shift are exact.)
__device__ __forceinline__ uint64_t sw128_kmajor_desc_at_row(uint32_t buf, uint32_t row) {
  return sw128_kmajor_desc(buf + row * 128u);
}

// Shared-memory matrix descriptor for an MN-major operand tile (the N index
// contiguous) stored with the 128-byte swizzle, as a TMA copy of 64 x 64
// boxes writes it: each box holds 64 consecutive N values (128 bytes) for
// each of 64 K rows, 8-row swizzle atoms 1024 bytes apart (the stride
// offset, along K); boxes of the next 64 N values follow 8192 bytes later
// (the leading offset, along N; a box of 128 K rows puts them 16384 bytes
// apart).  The tile base must be 1024-byte aligned; stepping K by 16 rows
// adds 2048 bytes, 128 in the start-address field.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr,
                                                      uint32_t n_block_bytes = 8192) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(n_block_bytes >> 4) << 16;     // leading offset: next 64 N
  d |= static_cast<uint64_t>(1024 >> 4) << 32;              // stride offset: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;                      // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                      // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with fp32 accumulation: A and B fp16
// (bf16 = false) or both bf16; A K-major, B K-major or (b_mn) MN-major.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool b_mn = false) {
  return (1u << 4)                              // D format: f32
         | ((bf16 ? 1u : 0u) << 7)              // A format
         | ((bf16 ? 1u : 0u) << 10)             // B format
         | ((b_mn ? 1u : 0u) << 16)             // B major: 0 K, 1 MN
         | (static_cast<uint32_t>(N >> 3) << 17)  // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24); // M / 16
}

// Warpgroup-wide register re-allocation (all 128 threads of a warpgroup
// execute it).  dec returns registers to the CTA's pool; inc waits until the
// pool can supply them.
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- globals
// Read-only loads: not volatile, so the compiler may hoist them above
// unrelated stores and keep several in flight.
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
__device__ __forceinline__ uint2 ldg_nc_v2(const void *p) {
  uint2 r;
  asm volatile("ld.global.nc.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
  return r;
}
// Bring the 128-byte lines of [p, p + bytes) into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void *p, int bytes) {
  const uintptr_t first = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(127);
  const uintptr_t last = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes) - 1;
  for (uintptr_t a = first; a <= last; a += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
}

// A load served from L2 (not a possibly stale L1 line): data another SM
// wrote in this launch.  Volatile, so it stays after the fence before it.
__device__ __forceinline__ uint4 ldcg_v4(const void *p) {
  uint4 r;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}

__device__ __forceinline__ void stg_v4(void *p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

}  // namespace fconv
