// The library's bounded mbarrier wait (csrc/iq_common.cuh) on the GPU, with no fault and no hang:
// a phase that nothing completes makes the wait give up after its limit and say so; a completed
// phase returns at once; the context stays usable afterwards.
#include <cstdio>

#include "../ggml_iq_codebook_accumulate_b300/csrc/iq_common.cuh"

__global__ void wait_once(int arrive, int *ok, unsigned long long *ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    iqk::mbar_init(&bar, 1);
    iqk::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (arrive) iqk::mbar_arrive(&bar);
    const uint64_t t0 = iqk::global_timer_ns();
    const bool done = iqk::mbar_wait_bounded(&bar, 0);
    *ns = iqk::global_timer_ns() - t0;
    *ok = done ? 1 : 0;
  }
}

static bool run(int arrive, int *d_ok, unsigned long long *d_ns, int &ok, unsigned long long &ns) {
  wait_once<<<1, 32>>>(arrive, d_ok, d_ns);
  if (cudaDeviceSynchronize() != cudaSuccess) return false;
  cudaMemcpy(&ok, d_ok, sizeof(int), cudaMemcpyDeviceToHost);
  cudaMemcpy(&ns, d_ns, sizeof(ns), cudaMemcpyDeviceToHost);
  return cudaGetLastError() == cudaSuccess;
}

int main() {
  int *d_ok;
  unsigned long long *d_ns;
  cudaMalloc(&d_ok, sizeof(int));
  cudaMalloc(&d_ns, sizeof(unsigned long long));
  int ok = -1;
  unsigned long long ns = 0;
  if (!run(0, d_ok, d_ns, ok, ns)) { printf("launch failed\n"); return 1; }
  printf("never-completed %d %llu %llu\n", ok, ns, iqk::kWaitLimitNs);
  if (!run(1, d_ok, d_ns, ok, ns)) { printf("launch failed\n"); return 1; }
  printf("completed %d %llu\n", ok, ns);
  return 0;
}
