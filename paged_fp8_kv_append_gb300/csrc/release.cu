// release.cu -- kv_release_pages: finished requests give their pages back.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section
// "Protecting a shared KV cache": a physical page's tag changes whenever the
// page is reallocated.  Releasing a request's pages and handing them out
// again (the append pops bump the tags) is what makes any mapping still
// recorded for them stale, and the tag check then aborts its user.
//
// The free list is a stack on the pool's free_list array: appends pop
// free_list[head++]; a release of T pages writes them, in (request, page)
// order, to free_list[head - T ...] and sets head -= T, so the next appends
// pop them back in that order.
//
// Kernel 1 (one CTA): the released-page count of every request, a block scan
// into the workspace, the checks (length, T <= head) and the head update.
// Kernel 2 (one CTA per request and chunk of 2048 pages): the scatter of
// those pages and the reset of that part of the page-table row.  Offsets live in the workspace, so kernel 2
// never reads a length another CTA is clearing.
#include "common.cuh"
#include "internal.h"

namespace kvfp8 {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kScatterThreads = 256;
constexpr int kScatterUnroll = 8;
constexpr int kScatterChunk = kScatterThreads * kScatterUnroll;  // pages per CTA

__device__ long long block_excl_scan(long long v, long long* warp_sums, long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[wid] = x;
  __syncthreads();
  if (wid == 0) {
    long long w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;
  }
  __syncthreads();
  const long long before = (wid > 0 ? warp_sums[wid - 1] : 0) + x - v;
  *total = warp_sums[(blockDim.x >> 5) - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kPlanThreads) release_plan_kernel(ReleaseArgs a) {
  pdl_wait();
  pdl_trigger();
  __shared__ long long warp_sums[32];
  __shared__ int s_bad;
  const long long P = a.d.page_size;
  long long* off = a.offsets;
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  long long carry = 0;
  for (int base = 0; base < a.B; base += kPlanThreads) {
    const int r = base + threadIdx.x;
    long long n = 0;
    if (r < a.B && (a.mask == nullptr || (a.mask[r] & a.mask_bits) != 0)) {
      const long long L = a.seq_lens[r];
      n = (L + P - 1) / P;
      if (L < 0 || n > a.max_pages) {
        s_bad = 1;
        n = 0;
      }
    }
    long long chunk;
    const long long before = block_excl_scan(n, warp_sums, &chunk);
    if (r < a.B) off[r] = carry + before;
    carry += chunk;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const long long head = a.d.ctl[KV_CTL_FREE_HEAD];
    const bool ok = !s_bad && head >= 0 && head <= a.d.num_pages && carry <= head;
    off[a.B] = carry;
    off[a.B + 1] = head - carry;  // first free-list slot written
    off[a.B + 2] = ok ? 1 : 0;
    if (ok)
      a.d.ctl[KV_CTL_FREE_HEAD] = (int32_t)(head - carry);
    else
      set_error(a.d.ctl, KV_ERR_INVALID_ARG);
  }
}

__global__ void __launch_bounds__(kScatterThreads) release_scatter_kernel(ReleaseArgs a) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const long long* off = a.offsets;
  if (off[a.B + 2] == 0) return;  // the plan refused the call
  if (a.mask != nullptr && (a.mask[r] & a.mask_bits) == 0) return;
  const long long o = off[r], n = off[r + 1] - o;
  const long long j0 = (long long)blockIdx.y * kScatterChunk;
  if (j0 >= n) {
    if (blockIdx.y == 0 && threadIdx.x == 0) a.seq_lens[r] = 0;  // owned no page
    return;
  }
  const long long base = off[a.B + 1] + o;
  int32_t* pt = a.page_table + (long long)r * a.max_pages;
  uint32_t* et = a.exp_tags + (long long)r * a.max_pages;
  int32_t p[kScatterUnroll];
#pragma unroll
  for (int i = 0; i < kScatterUnroll; ++i) {
    const long long j = j0 + i * kScatterThreads + threadIdx.x;
    p[i] = j < n ? pt[j] : 0;
  }
#pragma unroll
  for (int i = 0; i < kScatterUnroll; ++i) {
    const long long j = j0 + i * kScatterThreads + threadIdx.x;
    if (j < n) {
      a.d.free_list[base + j] = p[i];
      pt[j] = -1;
      et[j] = 0;
    }
  }
  if (blockIdx.y == 0 && threadIdx.x == 0) a.seq_lens[r] = 0;
}

}  // namespace

size_t release_ws_bytes(int B) { return sizeof(long long) * ((size_t)B + 3); }

cudaError_t launch_release(const ReleaseArgs& a, cudaStream_t s, int* launches) {
  cudaError_t e = launch_pdl(release_plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, a);
  if (e != cudaSuccess) return e;
  ++*launches;
  // one CTA per (request, chunk of 2048 pages of its page-table row)
  const unsigned chunks = (unsigned)((a.max_pages + kScatterChunk - 1) / kScatterChunk);
  e = launch_pdl(release_scatter_kernel, dim3((unsigned)a.B, chunks), dim3(kScatterThreads), 0, s,
                 a);
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace kvfp8
