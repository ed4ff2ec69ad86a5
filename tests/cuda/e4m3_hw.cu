// The GPU's own fp32 -> e4m3 conversion (round to nearest even, saturating to
// +-448: __nv_cvt_float_to_fp8 with __NV_SATFINITE) of a range of fp32 bit
// patterns.  Test infrastructure: built as a shared library and called by
// tests/test_oracle_e4m3_hw_gpu.py, which compares the oracle's encoder with
// it on all 2^32 patterns.  Shares nothing with the library or the oracle.
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

__global__ void convert(uint32_t first, uint32_t count, uint8_t* out) {
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    out[i] = (uint8_t)__nv_cvt_float_to_fp8(__uint_as_float(first + i), __NV_SATFINITE,
                                            __NV_E4M3);
}

uint8_t* g_buf = nullptr;
uint32_t g_cap = 0;

}  // namespace

// Codes of the fp32 patterns first, first + 1, ... (mod 2^32), count of them
// (count <= 2^30), into host_out.  Returns 0, or a nonzero CUDA failure code.
extern "C" int hw_e4m3_range(uint32_t first, uint32_t count, uint8_t* host_out) {
  if (count == 0) return 0;
  if (count > (1u << 30)) return -1;
  if (count > g_cap) {
    if (g_buf) cudaFree(g_buf);
    g_buf = nullptr;
    g_cap = 0;
    if (cudaMalloc(&g_buf, count) != cudaSuccess) return 1;
    g_cap = count;
  }
  convert<<<152 * 8, 256>>>(first, count, g_buf);
  if (cudaGetLastError() != cudaSuccess) return 2;
  if (cudaMemcpy(host_out, g_buf, count, cudaMemcpyDeviceToHost) != cudaSuccess) return 3;
  return 0;
}

extern "C" void hw_e4m3_free() {
  if (g_buf) cudaFree(g_buf);
  g_buf = nullptr;
  g_cap = 0;
}
