// Test-hook kernels: export the dropout keep mask and raw Philox blocks from
// the same device generator the attention kernels use.
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

// One thread per (row, 16-key group): keep[row][16g .. 16g+15].
__global__ void debug_dropout_kernel(uint8_t* keep, long long rows, int N, DropParams d) {
  const int groups = (N + 15) / 16;
  const long long total = rows * groups;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = t / groups;
    const int g = static_cast<int>(t % groups);
    const uint4 k = dropout_keep16(d, static_cast<uint32_t>(row), static_cast<uint32_t>(g));
    const uint32_t w[4] = {k.x, k.y, k.z, k.w};
    uint8_t* dst = keep + row * N + g * 16;
    for (int e = 0; e < 16 && g * 16 + e < N; ++e)
      dst[e] = ((w[e >> 2] >> (8 * (e & 3))) & 0xFFu) ? 1 : 0;
  }
}

__global__ void debug_philox_kernel(const uint4* ctr, uint4* out, int n, uint32_t k0, uint32_t k1) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n) out[t] = philox4x32_10(ctr[t], k0, k1);
}

}  // namespace

cudaError_t launch_debug_dropout(uint8_t* keep, int B, int H, int N, const DropParams& d,
                                 cudaStream_t stream) {
  const long long rows = static_cast<long long>(B) * H * N;
  debug_dropout_kernel<<<1024, 256, 0, stream>>>(keep, rows, N, d);
  return cudaGetLastError();
}

cudaError_t launch_debug_philox(const uint32_t* counters, uint32_t* out, int n, uint32_t k0,
                                uint32_t k1, cudaStream_t stream) {
  debug_philox_kernel<<<(n + 255) / 256, 256, 0, stream>>>(reinterpret_cast<const uint4*>(counters),
                                                           reinterpret_cast<uint4*>(out), n, k0, k1);
  return cudaGetLastError();
}

}  // namespace fa
