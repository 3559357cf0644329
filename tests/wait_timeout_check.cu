// A bounded mbarrier wait that nothing completes must give up after its time
// limit and report bit 0 in the status word, leaving the context usable.
// Built and run by tests/test_gpu_failure.py.
#include <cstdio>

#include "kvq_device.cuh"

__global__ void wait_never_completes(uint32_t* status, int* completed) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    kvq::mbar_init(&bar, 1);  // one arrival expected; none is ever made
    kvq::fence_mbar_init();
  }
  __syncthreads();
  const bool ok = kvq::mbar_wait_bounded(&bar, 0);
  if (threadIdx.x == 0) {
    if (!ok) kvq::report_timeout(status);
    *completed = ok ? 1 : 0;
  }
}

__global__ void add_one(int* x) { *x += 1; }

int main() {
  uint32_t* status = nullptr;
  int* completed = nullptr;
  if (cudaMalloc(&status, 4) != cudaSuccess || cudaMalloc(&completed, 4) != cudaSuccess) return 2;
  cudaMemset(status, 0, 4);
  cudaMemset(completed, 0, 4);
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  cudaEventRecord(e0);
  wait_never_completes<<<1, 32>>>(status, completed);
  cudaEventRecord(e1);
  cudaError_t err = cudaEventSynchronize(e1);
  float ms = 0.0f;
  cudaEventElapsedTime(&ms, e0, e1);
  uint32_t hs = 0;
  int hc = -1;
  cudaMemcpy(&hs, status, 4, cudaMemcpyDeviceToHost);
  cudaMemcpy(&hc, completed, 4, cudaMemcpyDeviceToHost);
  // the context must still run work afterwards
  add_one<<<1, 1>>>(completed);
  int after = -1;
  cudaError_t err2 = cudaMemcpy(&after, completed, 4, cudaMemcpyDeviceToHost);
  printf("status=%u completed=%d ms=%.1f err=%s after=%d err2=%s\n", hs, hc, ms, cudaGetErrorString(err), after,
         cudaGetErrorString(err2));
  return 0;
}
