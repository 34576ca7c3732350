// Quantisation for the FP8 forward: FA-3's FP8 with incoherent processing
// (cross-paper synthesis page on FlashAttention, section 2, the FA-3 entry).
// Q and K are multiplied by M = diag(signs) H / sqrt(d), H the Sylvester
// Hadamard matrix (orthogonal, so Q K^T is unchanged while outlier channels
// are spread over all d), then stored as e4m3 with a per-head scale
// amax / 448; V keeps its values and gets one scale per (head, column),
// applied to O's columns in the forward's epilogue. V is written transposed
// ([B*H, d, Np], Np = N rounded up to 16) so that the PV product reads it
// K-major like the other operands.
//
// Two passes over the inputs (both HBM-bound, one 128-row block of one head
// per CTA, one warp per row): the first finds the amaxes (atomicMax on the
// float bits, which order like the values for non-negative floats), the
// second rotates again, scales, converts (round to nearest even, saturating
// at 448) and writes the codes.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

namespace {

constexpr int kQuantThreads = 128;  // 4 warps, 32 rows each
constexpr float kE4m3Max = 448.0f;

// The four consecutive elements this lane holds of a 128-wide row
// (columns 4 lane .. 4 lane + 3), rotated: x <- (x * signs) H / sqrt(128).
// Sylvester's H is the fast Walsh-Hadamard transform: for each stride s the
// pair (i, i + s) inside each block of 2 s becomes (a + b, a - b). Strides 1
// and 2 are within the lane, 4 .. 64 across lanes (partner lane ^ (s / 4)).
__device__ __forceinline__ void hadamard128(float x[4], const float sg[4], bool on) {
  if (!on) return;  // no rotation requested: Q and K are quantised as they are
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < 4; ++t) x[t] *= sg[t];
  {
    const float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
    x[0] = a0 + a2;
    x[1] = a1 + a3;
    x[2] = a0 - a2;
    x[3] = a1 - a3;
  }
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float o = __shfl_xor_sync(0xffffffffu, x[t], m);
      x[t] = upper ? (o - x[t]) : (x[t] + o);
    }
  }
  const float inv = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int t = 0; t < 4; ++t) x[t] *= inv;
}

__device__ __forceinline__ void load4(const __nv_bfloat16* p, float x[4]) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  x[0] = __uint_as_float(w.x << 16);
  x[1] = __uint_as_float(w.x & 0xFFFF0000u);
  x[2] = __uint_as_float(w.y << 16);
  x[3] = __uint_as_float(w.y & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t e4m3x4(const float y[4]) {
  uint32_t c = 0;
#pragma unroll
  for (int t = 0; t < 4; ++t)
    c |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(y[t], __NV_SATFINITE, __NV_E4M3)) << (8 * t);
  return c;
}

__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? amax / kE4m3Max : 1.f; }

// amax[0 .. BH): |Q'|, [BH .. 2 BH): |K'|, [2 BH ..): |V| per (head, column).
__global__ void __launch_bounds__(kQuantThreads)
    fp8_amax_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const float* __restrict__ signs, int BH,
                    int N, unsigned int* __restrict__ amax) {
  constexpr int D = 128;
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ float vcol[4][D];
  __shared__ float red[2][4];
  const bool rot = signs != nullptr;
  float sg[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) sg[t] = rot ? signs[4 * lane + t] : 1.f;
  float mq = 0.f, mk = 0.f, mv[4] = {0.f, 0.f, 0.f, 0.f};
  for (int rr = warp; rr < kTile; rr += 4) {
    const int row = blk * kTile + rr;
    if (row >= N) break;
    const size_t off = (static_cast<size_t>(bh) * N + row) * D + 4 * lane;
    float x[4];
    load4(q + off, x);
    hadamard128(x, sg, rot);
#pragma unroll
    for (int t = 0; t < 4; ++t) mq = fmaxf(mq, fabsf(x[t]));
    load4(k + off, x);
    hadamard128(x, sg, rot);
#pragma unroll
    for (int t = 0; t < 4; ++t) mk = fmaxf(mk, fabsf(x[t]));
    load4(v + off, x);
#pragma unroll
    for (int t = 0; t < 4; ++t) mv[t] = fmaxf(mv[t], fabsf(x[t]));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) {
    mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, m));
    mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, m));
  }
  if (lane == 0) {
    red[0][warp] = mq;
    red[1][warp] = mk;
  }
#pragma unroll
  for (int t = 0; t < 4; ++t) vcol[warp][4 * lane + t] = mv[t];
  __syncthreads();
  if (threadIdx.x == 0) {
    const float a = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
    const float b = fmaxf(fmaxf(red[1][0], red[1][1]), fmaxf(red[1][2], red[1][3]));
    atomicMax(amax + bh, __float_as_uint(a));
    atomicMax(amax + BH + bh, __float_as_uint(b));
  }
  const int c = threadIdx.x;  // one column per thread (128 threads, d = 128)
  const float m = fmaxf(fmaxf(vcol[0][c], vcol[1][c]), fmaxf(vcol[2][c], vcol[3][c]));
  atomicMax(amax + 2 * BH + static_cast<size_t>(bh) * D + c, __float_as_uint(m));
}

__global__ void __launch_bounds__(kQuantThreads)
    fp8_quant_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, const float* __restrict__ signs, int BH,
                     int N, int Np, const unsigned int* __restrict__ amax,
                     uint8_t* __restrict__ q8, uint8_t* __restrict__ k8, uint8_t* __restrict__ vt8) {
  constexpr int D = 128;
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ __align__(16) uint8_t vt[D][kTile + 16];  // [column][row of the block], padded
  const bool rot = signs != nullptr;
  float sg[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) sg[t] = rot ? signs[4 * lane + t] : 1.f;
  const float iq = 1.f / scale_of(__uint_as_float(amax[bh]));
  const float ik = 1.f / scale_of(__uint_as_float(amax[BH + bh]));
  float iv[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    iv[t] = 1.f / scale_of(__uint_as_float(amax[2 * BH + static_cast<size_t>(bh) * D + 4 * lane + t]));
  for (int rr = warp; rr < kTile; rr += 4) {
    const int row = blk * kTile + rr;
    uint32_t cv = 0;
    if (row < N) {
      const size_t off = (static_cast<size_t>(bh) * N + row) * D + 4 * lane;
      float x[4];
      load4(q + off, x);
      hadamard128(x, sg, rot);
#pragma unroll
      for (int t = 0; t < 4; ++t) x[t] *= iq;
      *reinterpret_cast<uint32_t*>(q8 + off) = e4m3x4(x);
      load4(k + off, x);
      hadamard128(x, sg, rot);
#pragma unroll
      for (int t = 0; t < 4; ++t) x[t] *= ik;
      *reinterpret_cast<uint32_t*>(k8 + off) = e4m3x4(x);
      load4(v + off, x);
#pragma unroll
      for (int t = 0; t < 4; ++t) x[t] *= iv[t];
      cv = e4m3x4(x);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) vt[4 * lane + t][rr] = static_cast<uint8_t>(cv >> (8 * t));
  }
  __syncthreads();
  // V^T rows of this block: column c, keys blk*128 .. blk*128 + 127 (zeros past N),
  // written 16 bytes at a time up to the padded length Np.
  for (int i = threadIdx.x; i < D * (kTile / 16); i += kQuantThreads) {
    const int c = i / (kTile / 16), seg = i % (kTile / 16);
    const int key0 = blk * kTile + seg * 16;
    if (key0 >= Np) continue;
    const uint4 w = *reinterpret_cast<const uint4*>(&vt[c][seg * 16]);
    *reinterpret_cast<uint4*>(vt8 + (static_cast<size_t>(bh) * D + c) * Np + key0) = w;
  }
}

__global__ void fp8_scales_kernel(const unsigned int* __restrict__ amax, int BH,
                                  float* __restrict__ s_q, float* __restrict__ s_k,
                                  float* __restrict__ s_v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) {
    s_q[i] = scale_of(__uint_as_float(amax[i]));
    s_k[i] = scale_of(__uint_as_float(amax[BH + i]));
  }
  if (i < BH * 128) s_v[i] = scale_of(__uint_as_float(amax[2 * BH + i]));
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H;
  const dim3 grid((a.N + kTile - 1) / kTile, BH);
  cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(unsigned int) * static_cast<size_t>(BH) * 130,
                                  stream);
  if (e != cudaSuccess) return e;
  fp8_amax_kernel<<<grid, kQuantThreads, 0, stream>>>(a.q, a.k, a.v, a.signs, BH, a.N, a.amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_quant_kernel<<<grid, kQuantThreads, 0, stream>>>(a.q, a.k, a.v, a.signs, BH, a.N, a.Np,
                                                       a.amax, a.q8, a.k8, a.vt8);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_scales_kernel<<<(BH * 128 + 255) / 256, 256, 0, stream>>>(a.amax, BH, a.s_q, a.s_k, a.s_v);
  return cudaGetLastError();
}

}  // namespace fa
