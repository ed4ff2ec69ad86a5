// Exhaustive check of div_by_scale, div_fresh and the two-value quant_word_fresh
// (quant.cuh) against CUDA's
// correctly rounded division: for every bf16 bit pattern x and every scale the append
// kernels can produce (amax / 448 of a positive finite bf16 amax, and 1.0),
// the e4m3 code of the quotient must be the same.  Test infrastructure:
// built and run by tests/test_quant_exhaustive_gpu.py.  Prints the number of
// pairs checked and of mismatches, and the first mismatch if any.
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "quant.cuh"

__global__ void check(const float* scales, long long nscales, unsigned long long* bad,
                      unsigned long long* first) {
  const long long total = nscales << 16;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const float s = scales[i >> 16];
    const float x = kvfp8::bf16_bits_to_f32((uint32_t)(i & 0xFFFF));
    const float rs = __frcp_rn(s);
    const uint32_t ref = kvfp8::e4m3x2(__fdiv_rn(x, s), 0.0f) & 0xFFu;
    const uint32_t got = kvfp8::e4m3x2(kvfp8::div_by_scale(x, s, rs), 0.0f) & 0xFFu;
    // div_fresh serves a block's own rows (|x| <= its amax, so |x * rs| <=
    // 448 (1 + 2^-22)); checked here on the wider |x * rs| < 1024
    bool fresh_bad = false;
    if (kvfp8::scale_fast_ok(s) && fabsf(x * rs) < 1024.0f) {
      fresh_bad = (kvfp8::e4m3x2(kvfp8::div_fresh(x, s, rs), 0.0f) & 0xFFu) != ref;
      // the two-value word path on (x, -x): both codes
      const uint32_t b = (uint32_t)(i & 0xFFFF), nb = b ^ 0x8000u;
      const uint32_t ref_n = kvfp8::e4m3x2(__fdiv_rn(kvfp8::bf16_bits_to_f32(nb), s), 0.0f) & 0xFFu;
      const uint32_t pair = kvfp8::quant_word_fresh(b | (nb << 16), s, rs);
      fresh_bad = fresh_bad || (pair & 0xFFu) != ref || ((pair >> 8) & 0xFFu) != ref_n;
    }
    if (ref != got || fresh_bad) {
      atomicAdd(bad, 1ull);
      atomicMin(first, (unsigned long long)i);
    }
  }
}

int main() {
  // every scale amax/448 (IEEE fp32, as the device computes it) of a positive
  // finite bf16 amax; 1.0 stands for amax = 0 and for quotients that underflow
  std::vector<float> sc;
  sc.push_back(1.0f);
  for (uint32_t b = 1; b < 0x7F80u; ++b) {
    uint32_t u = b << 16;
    float a;
    memcpy(&a, &u, 4);
    const float q = a / 448.0f;  // IEEE fp32 division on the host
    if (q > 0.0f) sc.push_back(q);
  }
  std::sort(sc.begin(), sc.end());
  sc.erase(std::unique(sc.begin(), sc.end()), sc.end());
  float* d_sc;
  unsigned long long *d_bad, *d_first, h_bad = 0, h_first = ~0ull, init = ~0ull;
  if (cudaMalloc(&d_sc, sc.size() * 4) != cudaSuccess) return 2;
  cudaMalloc(&d_bad, 8);
  cudaMalloc(&d_first, 8);
  cudaMemcpy(d_sc, sc.data(), sc.size() * 4, cudaMemcpyHostToDevice);
  cudaMemset(d_bad, 0, 8);
  cudaMemcpy(d_first, &init, 8, cudaMemcpyHostToDevice);
  check<<<152 * 8, 256>>>(d_sc, (long long)sc.size(), d_bad, d_first);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    printf("cuda error\n");
    return 2;
  }
  cudaMemcpy(&h_bad, d_bad, 8, cudaMemcpyDeviceToHost);
  cudaMemcpy(&h_first, d_first, 8, cudaMemcpyDeviceToHost);
  printf("scales=%zu pairs=%llu mismatches=%llu\n", sc.size(),
         (unsigned long long)sc.size() << 16, h_bad);
  if (h_bad) {
    uint32_t xb = (uint32_t)(h_first & 0xFFFF);
    printf("first: x bits 0x%04x scale %.9g\n", xb, sc[h_first >> 16]);
  }
  return h_bad ? 1 : 0;
}
