// decode_plan.cuh -- the batch plan of decode attention, as one CTA of
// kDecodePlanThreads threads computes it.  Used by the plan kernel of the
// attention call and, inside the one-call step, by the append's plan kernel
// (which already knows every request's new length and abort bits), so that
// the step needs no separate plan launch.
#pragma once

#include <climits>

#include "common.cuh"
#include "internal.h"

namespace kvfp8 {

constexpr int kDecodePlanThreads = 1024;

// pfx[r] = exclusive prefix of units of work (pages) over requests that get
// output, and rq_skip.  A request is skipped (no pages, no output) when
// aborted or when its length is negative or needs more pages than its page
// table holds (that also sets KV_ERR_INVALID_ARG).
__device__ __forceinline__ void decode_plan_block(const DecodeArgs& a) {
  __shared__ int warp_sums[32];
  __shared__ int s_overflow;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int P = a.d.page_size;
  // the prefix is held in int32: a batch of more than 2^28 units (so that
  // units times head groups stay clear of 2^31; only possible with lengths no
  // pool can back) is refused as a whole
  long long carry = 0;
  if (threadIdx.x == 0) s_overflow = 0;
  for (int base = 0; base < a.B; base += kDecodePlanThreads) {
    const int r = base + threadIdx.x;
    int np = 0;
    if (r < a.B) {
      const long long L = a.seq_lens[r];  // 64-bit: L + P - 1 may pass 2^31
      const bool aborted = a.abort_mask != nullptr && a.abort_mask[r] != 0;
      const bool bad_len = L < 0 || (L + P - 1) / P > a.max_pages;
      if (!aborted && bad_len) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
      const bool skip = aborted || bad_len;
      // at most ceil(2^31 / P) units: an int
      np = skip ? 0 : (int)((L + a.unit_tokens - 1) / a.unit_tokens);
      a.ws.rq_skip[r] = skip ? 1 : 0;
    }
    int v = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[wid] = v;
    __syncthreads();
    if (wid == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += n;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (wid > 0 ? warp_sums[wid - 1] : 0);
    const long long excl = carry + incl - np;
    if (r < a.B) a.ws.pfx[r] = excl > INT_MAX ? INT_MAX : (int)excl;
    carry += warp_sums[31];
    __syncthreads();
  }
  if (carry > INT_MAX / 8) s_overflow = 1;  // same value in every thread
  __syncthreads();
  if (s_overflow) {  // nothing is attended; the call reports the batch
    for (int r = threadIdx.x; r <= a.B; r += kDecodePlanThreads) {
      a.ws.pfx[r] = 0;
      if (r < a.B) a.ws.rq_skip[r] = 1;
    }
    if (threadIdx.x == 0) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
    return;
  }
  if (threadIdx.x == 0) a.ws.pfx[a.B] = (int)carry;
}

// The same plan computed by one CTA of any size (a multiple of 32 threads, at
// most 1024) into shared memory, pfx_s[0 .. B] (B + 1 entries must fit), for
// a split kernel that plans its batch itself.  wsum: 32 ints of shared
// memory.  Every thread of the CTA must call it; returns (in every thread)
// whether the batch was refused (then nothing is attended).
__device__ __forceinline__ bool decode_plan_shared(const DecodeArgs& a, int32_t* pfx_s, int* wsum) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int P = a.d.page_size;
  if (a.B <= 32) {  // one warp scans the batch: no block-wide rounds
    if (wid == 0) {
      long long np = 0;
      if (lane < a.B) {
        const long long L = a.seq_lens[lane];
        const bool aborted = a.abort_mask != nullptr && a.abort_mask[lane] != 0;
        const bool bad_len = L < 0 || (L + P - 1) / P > a.max_pages;
        if (!aborted && bad_len) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
        np = (aborted || bad_len) ? 0 : (L + a.unit_tokens - 1) / a.unit_tokens;
      }
      long long v = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      const long long total = __shfl_sync(0xffffffffu, v, 31);
      // same refusal as decode_plan_block: more than 2^28 units attends nothing
      const bool refuse = total > INT_MAX / 8;
      if (lane < a.B) pfx_s[lane] = refuse ? 0 : (int)(v - np);
      if (lane == 0) {
        pfx_s[a.B] = refuse ? 0 : (int)total;
        wsum[0] = refuse ? 1 : 0;
        if (refuse) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
      }
    }
    __syncthreads();
    return wsum[0] != 0;
  }
  long long carry = 0;
  for (int base = 0; base < a.B; base += blockDim.x) {
    const int r = base + threadIdx.x;
    int np = 0;
    if (r < a.B) {
      const long long L = a.seq_lens[r];
      const bool aborted = a.abort_mask != nullptr && a.abort_mask[r] != 0;
      const bool bad_len = L < 0 || (L + P - 1) / P > a.max_pages;
      if (!aborted && bad_len) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
      np = (aborted || bad_len) ? 0 : (int)((L + a.unit_tokens - 1) / a.unit_tokens);
    }
    int v = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += n;
    }
    if (lane == 31) wsum[wid] = v;
    __syncthreads();
    long long before = carry;
    for (int k = 0; k < wid; ++k) before += wsum[k];
    long long chunk = 0;
    for (int k = 0; k < nw; ++k) chunk += wsum[k];
    const long long excl = before + v - np;
    if (r < a.B) pfx_s[r] = excl > INT_MAX ? INT_MAX : (int)excl;
    carry += chunk;
    __syncthreads();
  }
  // same refusal as decode_plan_block: more than 2^28 units attends nothing
  const bool refuse = carry > INT_MAX / 8;
  if (refuse) {
    for (int r = threadIdx.x; r <= a.B; r += blockDim.x) pfx_s[r] = 0;
    if (threadIdx.x == 0) set_error(a.d.ctl, KV_ERR_INVALID_ARG);
  } else if (threadIdx.x == 0) {
    pfx_s[a.B] = (int)carry;
  }
  __syncthreads();
  return refuse;
}

// The plan of decode_plan_shared stored into the workspace for the combine
// kernel (pfx and rq_skip, as decode_plan_block writes them); one CTA.
static __device__ __noinline__ void decode_plan_store(const DecodeArgs& a, const int32_t* pfx_s,
                                               bool refused) {
  const int P = a.d.page_size;
  for (int r = threadIdx.x; r <= a.B; r += blockDim.x) {
    a.ws.pfx[r] = pfx_s[r];
    if (r < a.B) {
      const long long L = a.seq_lens[r];
      const bool aborted = a.abort_mask != nullptr && a.abort_mask[r] != 0;
      const bool bad_len = L < 0 || (L + P - 1) / P > a.max_pages;
      a.ws.rq_skip[r] = (refused || aborted || bad_len) ? 1 : 0;
    }
  }
}

}  // namespace kvfp8
