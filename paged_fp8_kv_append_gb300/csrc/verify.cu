// verify.cu -- kv_verify_tags: the batched page-tag integrity check.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Protecting a shared KV cache": each request's recorded (page, tag) list is
// checked against the physical tags before decode reads the cache; any
// mismatch aborts that request.  The post runs the check as its own batched
// pass rather than inside the attention kernel, which would race between
// thread groups; so does this library.
//
// One cluster of 8 CTAs per request, each CTA taking an eighth of the
// request's pages, so a long request's random tag gathers are spread over 8
// SMs.  Each thread issues all of its page-table and expected-tag loads before
// the dependent tag gathers; the CTAs' results are OR-ed through distributed
// shared memory and the cluster's first CTA writes the mask byte.
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

namespace cg = cooperative_groups;

constexpr int kCluster = 8;
constexpr int kThreads = 128;
constexpr int kUnroll = 16;

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    verify_kernel(VerifyArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ int cta_bad;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int r = blockIdx.x / kCluster;
  const long long L = a.seq_lens[r];
  const long long n = (L + a.page_size - 1) / a.page_size;
  int bad = 0;
  if (L < 0 || n > a.max_pages) {
    bad = 1;
  } else {
    const long long per = (n + kCluster - 1) / kCluster;
    const long long j0 = (long long)rank * per, j1 = min(n, j0 + per);
    const int32_t* pt = a.page_table + (long long)r * a.max_pages;
    const uint32_t* et = a.exp_tags + (long long)r * a.max_pages;
    for (long long base = j0; base < j1; base += (long long)kThreads * kUnroll) {
      int p[kUnroll];
      uint32_t e[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long j = base + (long long)u * kThreads + threadIdx.x;
        p[u] = 0;
        e[u] = 0;
        if (j < j1) {
          p[u] = __ldg(pt + j);
          e[u] = __ldg(et + j);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long j = base + (long long)u * kThreads + threadIdx.x;
        if (j < j1) {
          if (p[u] < 0 || p[u] >= a.num_pages)
            bad = 1;
          else if (a.tags[p[u]] != e[u])
            bad = 1;
        }
      }
    }
  }
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) cta_bad = bad;
  cluster.sync();
  if (rank == 0 && threadIdx.x == 0) {
    int any = 0;
    for (int k = 0; k < kCluster; ++k) any |= *cluster.map_shared_rank(&cta_bad, k);
    a.abort_mask[r] = any ? 1 : 0;
  }
  cluster.sync();  // every CTA's flag stays readable until the first CTA is done
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t s, int* launches) {
  if (a.B <= 0) return cudaSuccess;
  const cudaError_t e =
      launch_pdl(verify_kernel, dim3((unsigned)a.B * kCluster), dim3(kThreads), 0, s, a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
