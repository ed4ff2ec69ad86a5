// The bounded wait every in-kernel hand-off of the library uses (mbar_wait,
// common.cuh), run on a barrier that nothing ever arrives on: it must give up
// after its limit, return false, record KV_ERR_TIMEOUT and the caller's
// location word in the control block, and make the other waiting warps give
// up at once through the shared abort flag -- so a lost arrival becomes an
// error code and the context stays usable.  A barrier that does complete is
// waited on normally.  Test infrastructure: built and run by
// tests/test_wait_timeout_gpu.py.
#include <cuda_runtime.h>
#include <stdio.h>

#include "common.cuh"

__global__ void waiters(int32_t* ctl, unsigned long long* out) {
  __shared__ uint64_t never, done;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    kvfp8::mbar_init(&never, 1);
    kvfp8::mbar_init(&done, 1);
    abort_flag = 0;
    kvfp8::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {  // a phase that completes
    if (lane == 0) kvfp8::mbar_arrive(&done);
    const bool ok = kvfp8::mbar_wait(&done, 0, &abort_flag, ctl, 0x111);
    if (lane == 0) out[0] = ok ? 1 : 0;
  }
  __syncthreads();
  // every warp waits for a phase that never completes
  const uint64_t t0 = kvfp8::global_ns();
  const bool ok = kvfp8::mbar_wait(&never, 0, &abort_flag, ctl, 0x200 + warp);
  const uint64_t t1 = kvfp8::global_ns();
  if (lane == 0) {
    out[1 + 2 * warp] = ok ? 1 : 0;
    out[2 + 2 * warp] = t1 - t0;
  }
}

int main() {
  int32_t* ctl;
  unsigned long long* out;
  unsigned long long h[1 + 2 * 4];
  int32_t hc[KV_CTL_WORDS];
  if (cudaMalloc(&ctl, sizeof(hc)) != cudaSuccess) return 2;
  if (cudaMalloc(&out, sizeof(h)) != cudaSuccess) return 2;
  cudaMemset(ctl, 0, sizeof(hc));
  cudaMemset(out, 0xFF, sizeof(h));
  waiters<<<1, 128>>>(ctl, out);
  if (cudaDeviceSynchronize() != cudaSuccess) {
    printf("cuda error\n");
    return 2;
  }
  cudaMemcpy(h, out, sizeof(h), cudaMemcpyDeviceToHost);
  cudaMemcpy(hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost);
  // the context is still usable: a second launch of the same kernel on a
  // fresh control block behaves the same way
  printf("completed_wait=%llu error=%d wait_info=0x%x\n", h[0], hc[KV_CTL_ERROR],
         (unsigned)hc[KV_CTL_WAIT_INFO]);
  for (int w = 0; w < 4; ++w)
    printf("warp %d: ok=%llu waited_ms=%.1f\n", w, h[1 + 2 * w], h[2 + 2 * w] / 1e6);
  int bad = 0;
  if (h[0] != 1) bad = 1;
  if (hc[KV_CTL_ERROR] != KV_ERR_TIMEOUT) bad = 1;
  if (hc[KV_CTL_WAIT_INFO] < 0x200 || hc[KV_CTL_WAIT_INFO] > 0x203) bad = 1;
  for (int w = 0; w < 4; ++w)
    if (h[1 + 2 * w] != 0 || h[2 + 2 * w] > 4000000000ull) bad = 1;
  unsigned long long longest = 0;
  for (int w = 0; w < 4; ++w) longest = h[2 + 2 * w] > longest ? h[2 + 2 * w] : longest;
  if (longest < kvfp8::kWaitLimitNs) bad = 1;
  cudaMemset(ctl, 0, sizeof(hc));
  waiters<<<1, 128>>>(ctl, out);
  if (cudaDeviceSynchronize() != cudaSuccess) bad = 1;
  cudaMemcpy(hc, ctl, sizeof(hc), cudaMemcpyDeviceToHost);
  if (hc[KV_CTL_ERROR] != KV_ERR_TIMEOUT) bad = 1;
  printf("second launch error=%d\n%s\n", hc[KV_CTL_ERROR], bad ? "FAIL" : "PASS");
  return bad;
}
