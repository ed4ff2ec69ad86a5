// common.cuh -- device helpers shared by the kernels of the paged FP8 KV
// library: error word, bounded mbarrier waits, bulk (TMA) copies, small
// reductions.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvfp8.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library targets sm_103a (Blackwell) only"
#endif

namespace kvfp8 {

// ---------------------------------------------------------------- errors

// First device-side error wins; later errors leave the word unchanged.
__device__ __forceinline__ void set_error(int32_t* ctl, int code) {
  atomicCAS(reinterpret_cast<int*>(ctl + KV_CTL_ERROR), 0, code);
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any single wait inside a kernel.  Every legitimate wait in
// this library is a producer/consumer hand-off inside one CTA that completes
// in microseconds; this bound only turns a bug into an error code instead of
// a hung GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ------------------------------------------------------------- mbarriers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// One bounded probe of phase `parity`.  The suspend-time hint lets the
// hardware park the waiting warp until the phase completes (or the hint
// elapses) instead of spinning, so waiting warps leave the issue slots to the
// warps doing work.
constexpr uint32_t kSuspendHintNs = 1000000u;  // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false)
// when *abort_flag (shared memory) is set by another warp or after
// kWaitLimitNs, in which case it sets the abort flag, KV_ERR_TIMEOUT and (first
// timeout wins) the diagnostic word ctl[KV_CTL_WAIT_INFO] = `info`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, int32_t* ctl,
                                          int info = 0) {
  if (*abort_flag) return false;  // once a wait has given up, nothing waits any more
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        if (atomicCAS(reinterpret_cast<int*>(ctl + KV_CTL_ERROR), 0, KV_ERR_TIMEOUT) == 0)
          ctl[KV_CTL_WAIT_INFO] = info;
        return false;
      }
    }
  }
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation and waits for the grids before it (with
// their memory visible) before its first global-memory access, so the order
// of the stream is kept exactly while a kernel's launch overlaps the tail of
// the previous one.  `trigger` lets the next kernel launch early (its CTAs
// then sit in its own wait).  Every kernel triggers right after its own wait,
// so a kernel's dependents launch only once the kernel before it has
// completed: at most two grids of the stream are resident at a time.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Diagnostic word of a wait (see KV_CTL_WAIT_INFO).
__device__ __forceinline__ int wait_info(int warp, int which, int stage) {
  return (int)((blockIdx.x << 12) | ((warp & 31) << 7) | ((which & 1) << 6) | (stage & 63));
}

// ------------------------------------------------------ bulk (TMA) copies

// Non-tensor bulk copy global -> shared, completion counted in bytes on
// `bar`.  Both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once per call (the streamed KV pages).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// -------------------------------------------------------------- misc

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace kvfp8
