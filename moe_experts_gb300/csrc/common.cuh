// Shared device/host helpers of the epq CUDA library (sm_103a).
//
// Device side: mbarrier + 1-D bulk-copy (TMA engine) pipeline primitives with
// bounded waits, programmatic-dependent-launch controls, fp16 decoding and
// small warp reductions.  Host side: status plumbing and a per-device
// attribute cache.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "epq.h"

namespace epq {

// ------------------------------------------------------------------ errors
// Device-side error record (one word per device, defined in api.cu and
// passed to every kernel as a pointer).  A kernel whose pipeline wait runs
// past its time limit writes a code there and returns instead of spinning on.
enum DeviceError : unsigned {
  DEVERR_NONE = 0,
  DEVERR_FULL_WAIT = 1,    // consumer waited too long for a tile
  DEVERR_EMPTY_WAIT = 2,   // producer waited too long for a free stage
  DEVERR_DRAIN_WAIT = 3,   // copies still in flight at exit
  DEVERR_RED_WAIT = 4,     // waited too long for the cross-warp reduction
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// A waiting thread is suspended until the phase completes or kSuspendNs
// pass, whichever is first, so waiters do not take issue slots from the
// warps that work.
constexpr uint32_t kSuspendNs = 100000;  // 100 us

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// The same test without the suspend hint: the thread polls (for waits that
// are usually short and on the critical path of every thread of the CTA).
__device__ __forceinline__ bool mbar_test_poll(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Time limit of every pipeline wait.  A correct pipeline never comes close:
// the longest legitimate wait is one tile copy behind a busy HBM.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// Record the first timeout of the device: err[0] = code, err[1] = block,
// err[2] = `where` (the pipeline step, e.g. tile index), err[3] = thread.
__device__ __forceinline__ void record_error(unsigned *err, unsigned code, unsigned where) {
  if (atomicCAS(err, 0u, code) == 0u) {
    err[1] = blockIdx.x;
    err[2] = where;
    err[3] = threadIdx.x;
    __threadfence();
  }
}

// Bounded parity wait.  Returns false (after recording `code`) on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err, unsigned code,
                                          unsigned where = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, code, where);
      return false;
    }
  }
}

// Bounded parity wait that polls without suspending.
__device__ __forceinline__ bool mbar_wait_poll(uint64_t *bar, uint32_t parity, unsigned *err, unsigned code,
                                               unsigned where = 0) {
  if (mbar_test_poll(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_test_poll(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(err, code, where);
      return false;
    }
  }
}

// Warp-uniform bounded wait: lane 0 spins (bounded), the outcome is broadcast,
// and on success every lane performs its own acquire of the completed phase
// (which returns at once).  All lanes of the warp must call it.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, unsigned *err, unsigned code,
                                          unsigned where = 0) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, err, code, where) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) ok = mbar_wait(bar, parity, err, code, where) ? 1 : 0;
  return __all_sync(0xffffffffu, ok) != 0;
}

// warp_wait that polls without suspending.
__device__ __forceinline__ bool warp_wait_poll(uint64_t *bar, uint32_t parity, unsigned *err, unsigned code,
                                               unsigned where = 0) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait_poll(bar, parity, err, code, where) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (ok) ok = mbar_wait_poll(bar, parity, err, code, where) ? 1 : 0;
  return __all_sync(0xffffffffu, ok) != 0;
}

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar`
// (bytes and both addresses must be multiples of 16).
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bring the 128-byte line holding `p` into this SM's L1 (no register result).
__device__ __forceinline__ void prefetch_l1(const void *p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Programmatic dependent launch: wait for the preceding kernel's writes /
// allow the next kernel to begin its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier over `nthreads` threads (id 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_sync(unsigned id, unsigned nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------------ math helpers
__device__ __forceinline__ float half_bits_to_float(uint32_t h16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h16 & 0xFFFFu)));
}

// Exact power of two 2^e for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// x * 2^e for any e where the result is a normal float (two exact steps).
__device__ __forceinline__ float scale_pow2(float x, int e) {
  int e1 = e / 2;
  return x * exp2i(e1) * exp2i(e - e1);
}

// Packed float32x2 fused multiply-add (sm_100+): (d0,d1) += (a0,a1)*(b0,b1),
// IEEE round-to-nearest, subnormals preserved.
__device__ __forceinline__ void ffma2(float &d0, float &d1, float a0, float a1, float b0, float b1) {
  uint64_t a, b, c;
  asm("mov.b64 %0, {%1,%2};" : "=l"(a) : "f"(a0), "f"(a1));
  asm("mov.b64 %0, {%1,%2};" : "=l"(b) : "f"(b0), "f"(b1));
  asm("mov.b64 %0, {%1,%2};" : "=l"(c) : "f"(d0), "f"(d1));
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(a), "l"(b));
  asm("mov.b64 {%0,%1}, %2;" : "=f"(d0), "=f"(d1) : "l"(c));
}

template <int W>
__device__ __forceinline__ float warp_sum_xor(float v) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Largest of the warp's non-negative values (NaN counts as 0) in one
// redux.sync: non-negative floats order like their bit patterns.
__device__ __forceinline__ float warp_absmax(float v) {
  return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fmaxf(v, 0.0f))));
}

__device__ __forceinline__ float warp_min_all(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace epq

// ------------------------------------------------------------------ host side
namespace epq {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int major = 0, minor = 0;
  int max_smem_optin = 0;
  int l2_bytes = 0;
};

// Attributes of the current device (cached per device).  Returns false when
// no device is current or the query fails.
bool current_device(DeviceInfo *out);

// Device address of the error word of the current device (looked up once
// per device with cudaGetSymbolAddress), or nullptr on failure.
unsigned *device_error_slot();

// Current tuning values (see epq_set_tuning).
int tune_tile_bytes();
int tune_ring_bytes();
// 0 = automatic, 1 = CUDA-core engines only, 2 = tensor-core engine where it applies
int tune_gemv_engine();
// stages a tensor-core GEMV issues before its grid-dependency wait (weights_ready)
int tune_early_stages();
// k-parts (warps per 8-row block) of the tensor-core GEMV, 0 = chosen by shape
int tune_tc_split();
// most key/value rows of one attention copy chunk, 0 = as many as fit
int tune_attn_chunk();
// most superblocks of x operands per chunk of the vector-column GEMV, 0 = as many as fit
int tune_vn_chunk();
// CTAs per cluster of the vector-column GEMV (1, 2, 4), 0 = automatic
int tune_vn_cluster();

// Record a CUDA error for epq_last_cuda_error() and return EPQ_ERR_CUDA.
epq_status cuda_fail(cudaError_t e);

// Map the result of cudaGetLastError() after a launch.
inline epq_status check_launch() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? EPQ_OK : cuda_fail(e);
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch with the programmatic-stream-serialization attribute so that the
// kernel may start while the previous kernel on the stream drains; the
// kernel itself calls pdl_wait() before reading data produced upstream.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace epq
