// Test helper: raw Philox4x32-10 blocks from cuRAND's device generator, used
// to pin the oracle's Philox implementation to an external one.
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_kernel.h>

__global__ void curand_blocks_kernel(uint4* out, int n, unsigned long long seed,
                                     unsigned long long subsequence, unsigned long long skip) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  curandStatePhilox4_32_10_t st;
  curand_init(seed, subsequence, skip, &st);
  for (int t = 0; t < n; ++t) out[t] = curand4(&st);
}

// out: device uint32 [n][4]. Generator state: key = seed, counter high words =
// subsequence (= offset), counter word 1 = row (skip of 4 * (row << 32) outputs).
extern "C" int curand_philox_blocks(void* out, int n, unsigned long long seed,
                                    unsigned long long offset, unsigned int row, unsigned int) {
  const unsigned long long skip = 4ull * (static_cast<unsigned long long>(row) << 32);
  curand_blocks_kernel<<<1, 1>>>(static_cast<uint4*>(out), n, seed, offset, skip);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
