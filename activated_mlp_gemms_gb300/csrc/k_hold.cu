// k_hold -- a testing kernel that keeps SMs busy for a given time, so that
// tests can run the GEMMs while only part of their grid is resident.  Each
// CTA takes HOLD_SMEM_BYTES of shared memory (more than a GEMM CTA leaves
// free on its SM) and spins on the global timer until the time is up.  It
// reads and writes no global memory and waits on nothing else.
#include "gemm_params.h"
#include "ptx.cuh"

namespace mlpk {

__global__ void __launch_bounds__(32) k_hold(unsigned long long ns) {
  extern __shared__ uint8_t hold_smem[];
  const uint64_t t0 = globaltimer_ns();
  // at most 2^26 polls, whatever the timer reads
  for (uint32_t n = 0; n < (1u << 26); ++n) {
    if (globaltimer_ns() - t0 >= ns) break;
    __nanosleep(1000);
  }
  if (threadIdx.x == 0) hold_smem[0] = 0;  // the allocation is the point; nothing reads it
}

cudaError_t launch_hold(int ctas, unsigned long long ns, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(k_hold, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       HOLD_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  k_hold<<<ctas, 32, HOLD_SMEM_BYTES, stream>>>(ns);
  return cudaGetLastError();
}

}  // namespace mlpk
