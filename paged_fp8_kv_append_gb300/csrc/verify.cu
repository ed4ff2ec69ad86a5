// verify.cu -- kv_verify_tags: the batched page-tag integrity check.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Protecting a shared KV cache": each request's recorded (page, tag) list is
// checked against the physical tags before decode reads the cache; any
// mismatch aborts that request.  The post runs the check as its own batched
// pass rather than inside the attention kernel, which would race between
// thread groups; so does this library.
//
// One CTA per request.  Each thread issues all of its page-table and
// expected-tag loads before the dependent tag gathers, so a request of up to
// kThreads * kUnroll pages costs two memory round trips.
#include "common.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

constexpr int kThreads = 1024;
constexpr int kUnroll = 16;

__global__ void __launch_bounds__(kThreads) verify_kernel(VerifyArgs a) {
  const int r = blockIdx.x;
  const long long L = a.seq_lens[r];
  const long long n = (L + a.page_size - 1) / a.page_size;
  int bad = 0;
  if (L < 0 || n > a.max_pages) {
    bad = 1;
  } else {
    const int32_t* pt = a.page_table + (long long)r * a.max_pages;
    const uint32_t* et = a.exp_tags + (long long)r * a.max_pages;
    for (long long base = 0; base < n; base += (long long)kThreads * kUnroll) {
      int p[kUnroll];
      uint32_t e[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long j = base + (long long)u * kThreads + threadIdx.x;
        p[u] = 0;
        e[u] = 0;
        if (j < n) {
          p[u] = __ldg(pt + j);
          e[u] = __ldg(et + j);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long j = base + (long long)u * kThreads + threadIdx.x;
        if (j < n) {
          if (p[u] < 0 || p[u] >= a.num_pages)
            bad = 1;
          else if (a.tags[p[u]] != e[u])
            bad = 1;
        }
      }
    }
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) a.abort_mask[r] = bad ? 1 : 0;
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s, int* launches) {
  if (a.B <= 0) return cudaSuccess;
  verify_kernel<<<a.B, kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
