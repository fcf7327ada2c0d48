// hold_sms.cu -- a test helper, not part of libep: a kernel that keeps SMs
// busy for a fixed time and then returns on its own, so a test can run a
// dispatch while another stream holds part (or all) of the GPU.
//
// Each CTA takes `smem_bytes` of dynamic shared memory (enough that a
// dispatch CTA cannot share its SM) and waits on %globaltimer until `ns`
// nanoseconds have passed since it started.  The loop is also capped by an
// iteration count, so it ends even if the timer were to stand still.

#include <cstdint>

#include <cuda_runtime.h>

__global__ void hold_sm_kernel(unsigned long long ns) {
  extern __shared__ unsigned char pad[];
  unsigned long long t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  if (threadIdx.x == 0) pad[0] = 1;
  for (long long it = 0; it < 20000000LL; ++it) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    if (t - t0 >= ns) break;
    __nanosleep(500);
  }
}

extern "C" int hold_sms(int ctas, int smem_bytes, long long ns, void* stream) {
  if (ctas <= 0 || smem_bytes < 0 || ns < 0 || ns > 1000000000LL) return 1;
  if (cudaFuncSetAttribute(hold_sm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_bytes) != cudaSuccess)
    return 2;
  hold_sm_kernel<<<ctas, 128, smem_bytes, static_cast<cudaStream_t>(stream)>>>(
      (unsigned long long)ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
