// Latency probe of the die-aware placement.  One CTA runs on every SM (the
// dynamic shared memory keeps it alone there) and times chains of dependent
// L2 loads to each 128-byte line of a semaphore pool.  The host clusters the
// SMs by these latency vectors into the two dies and gives each line the die
// whose SMs reach it faster (place.cpp).
#include <cuda_runtime.h>

#include "kernels.h"

namespace dash {
namespace {

constexpr int kProbeReps = 2;
constexpr int kProbeChain = 4;

// the first word of every line holds its own word index
__global__ void probe_selfidx(unsigned *pool, int n_lines) {
  const int a = blockIdx.x * blockDim.x + threadIdx.x;
  if (a < n_lines) pool[(size_t)a * 32] = (unsigned)a * 32u;
}

// lat[cta][line]: the shortest of kProbeReps chains of kProbeChain dependent
// loads (each load's address is the previous load's value, and a shared-memory
// store of each value keeps the clock read behind the last load), per load.
__global__ void __launch_bounds__(32) probe_homes(const unsigned *pool, int n_lines, unsigned *lat, int *smid_out) {
  __shared__ unsigned sink[kProbeChain];
  if (threadIdx.x != 0) return;
  unsigned sm;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
  smid_out[blockIdx.x] = (int)sm;
  const unsigned limit = (unsigned)n_lines * 32u;
  for (int a = 0; a < n_lines; ++a) {
    unsigned best = 0xffffffffu;
    for (int rep = 0; rep < kProbeReps; ++rep) {
      unsigned j = (unsigned)a * 32u;
      const long long t0 = clock64();
#pragma unroll
      for (int k = 0; k < kProbeChain; ++k) {
        unsigned v;
        asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(pool + j) : "memory");
        asm volatile("st.shared.u32 [%0], %1;" ::"r"((unsigned)__cvta_generic_to_shared(&sink[k])), "r"(v)
                     : "memory");
        j = v < limit ? v : 0u;  // the pool holds only self indices; stay inside it regardless
      }
      const unsigned d = (unsigned)((clock64() - t0) / kProbeChain);
      best = d < best ? d : best;
    }
    lat[(size_t)blockIdx.x * n_lines + a] = best;
  }
}

}  // namespace

cudaError_t launch_probe_homes(unsigned *pool, int n_lines, unsigned *lat, int *smid_out, int num_sms,
                               cudaStream_t stream) {
  probe_selfidx<<<(n_lines + 255) / 256, 256, 0, stream>>>(pool, n_lines);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(probe_homes, cudaFuncAttributeMaxDynamicSharedMemorySize, kMinSmemOneCtaPerSm);
  if (e != cudaSuccess) return e;
  probe_homes<<<num_sms, 32, kMinSmemOneCtaPerSm, stream>>>(pool, n_lines, lat, smid_out);
  return cudaGetLastError();
}

}  // namespace dash
