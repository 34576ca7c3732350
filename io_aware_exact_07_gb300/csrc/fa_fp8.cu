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
// Two passes over the inputs, both HBM-bound: the first finds the amaxes
// (atomicMax on the float bits, which order like the values for non-negative
// floats), the second rotates again, scales, converts (round to nearest even,
// saturating at 448) and writes the codes. One CTA takes a 128-row block of one
// head; half a warp takes one 128-column row, each lane 8 consecutive columns
// (16-byte loads), and a lane issues the Q, K and V loads of its next two rows
// before it rotates any of them, so that enough bytes are in flight to cover
// the memory latency. With grouped K/V heads (Hkv < H) the grid runs over the
// B*H query heads and the CTAs of head index bh < B*Hkv also take K/V head bh;
// the test is uniform over a CTA.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"
#include "fa_fp8.h"

namespace fa {

namespace {

constexpr int kQuantThreads = 256;  // 8 warps = 16 half-warps, one row each at a time
constexpr int kQuantRowsPerIter = 4 * (kQuantThreads / 32);  // two rows per half-warp in flight
constexpr float kE4m3Max = 448.0f;

// The eight consecutive elements this lane holds of a 128-wide row (columns
// 8 l .. 8 l + 7, l = lane mod 16), rotated and scaled: x <- ((x * f) H),
// f[t] = signs[8 l + t] / sqrt(128) times the code scale's inverse, which is
// the same as (x * signs) H / sqrt(128) / scale since H is linear.
// Sylvester's H is the fast Walsh-Hadamard transform: for each stride s the
// pair (i, i + s) inside each block of 2 s becomes (a + b, a - b). Strides 1, 2
// and 4 are within the lane, 8 .. 64 across the lanes of the half-warp (partner
// lane ^ (s / 8), one fused multiply-add: the lower lane adds, the upper one
// subtracts its own value from the partner's); the stages commute.
__device__ __forceinline__ void hadamard128(float x[8], const float f[8]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int t = 0; t < 8; ++t) x[t] *= f[t];
#pragma unroll
  for (int s = 1; s < 8; s <<= 1)
#pragma unroll
    for (int t = 0; t < 8; ++t)
      if ((t & s) == 0) {
        const float a = x[t], b = x[t + s];
        x[t] = a + b;
        x[t + s] = a - b;
      }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const float self = (lane & m) != 0 ? -1.f : 1.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) x[t] = fmaf(self, x[t], __shfl_xor_sync(0xffffffffu, x[t], m));
  }
}

__device__ __forceinline__ uint4 load8(const __nv_bfloat16* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));  // read once per pass: evict first
}

__device__ __forceinline__ void unpack8(const uint4 w, float x[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    x[2 * t] = __uint_as_float(u[t] << 16);
    x[2 * t + 1] = __uint_as_float(u[t] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

__device__ __forceinline__ uint2 e4m3x8(const float y[8]) {
  return make_uint2(e4m3x4(y[0], y[1], y[2], y[3]), e4m3x4(y[4], y[5], y[6], y[7]));
}

__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? amax / kE4m3Max : 1.f; }

// V^T staging in shared memory: column c of the block holds its 128 key bytes
// as 32 words, word g stored at position g ^ vt_swz(c). The byte stores (the 16
// lanes of a half-warp write one row into columns 8 l + t) and the 16-byte
// read-out (a warp reads 8 segments of 4 columns) then each touch 32 distinct
// banks: bits 3..6 of c move the word by up to 30, bits 0..1 by up to 3.
__device__ __forceinline__ int vt_swz(int c) { return (c & 3) ^ (((c >> 3) & 15) << 1); }

// amax[0 .. BH): |Q'| per query head, [BH .. BH + BHkv): |K'| per K/V head,
// [BH + BHkv ..): |V| per (K/V head, column).
__global__ void __launch_bounds__(kQuantThreads)
    fp8_amax_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const float* __restrict__ signs, int BH,
                    int BHkv, int N, unsigned int* __restrict__ amax) {
  constexpr int D = 128;
  constexpr int kWarps = kQuantThreads / 32;
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = 2 * warp + (lane >> 4), col = 8 * (lane & 15);  // half-warp, first column
  __shared__ float vcol[2 * kWarps][D];
  __shared__ float red[2][kWarps];
  const bool rot = signs != nullptr;
  const bool has_kv = bh < BHkv;
  constexpr float kInvSqrt = 0.08838834764831845f;  // 1 / sqrt(128)
  float f[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) f[t] = rot ? signs[col + t] * kInvSqrt : 1.f;
  float mq = 0.f, mk = 0.f, mv[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) mv[t] = 0.f;
  const int rows = min(kTile, N - blk * kTile);
  for (int r0 = 0; r0 < rows; r0 += kQuantRowsPerIter) {
    uint4 wq[2], wk[2], wv[2];
    bool in[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // all loads of both rows first
      const int rr = r0 + hw + u * (2 * kWarps);
      in[u] = rr < rows;
      const size_t off = (static_cast<size_t>(bh) * N + blk * kTile + rr) * D + col;
      wq[u] = in[u] ? load8(q + off) : make_uint4(0, 0, 0, 0);
      wk[u] = in[u] && has_kv ? load8(k + off) : make_uint4(0, 0, 0, 0);
      wv[u] = in[u] && has_kv ? load8(v + off) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // rows past the end hold zeros, which change no maximum
      float x[8];
      unpack8(wq[u], x);
      if (rot) hadamard128(x, f);
#pragma unroll
      for (int t = 0; t < 8; ++t) mq = fmaxf(mq, fabsf(x[t]));
      unpack8(wk[u], x);
      if (rot) hadamard128(x, f);
#pragma unroll
      for (int t = 0; t < 8; ++t) mk = fmaxf(mk, fabsf(x[t]));
      unpack8(wv[u], x);
#pragma unroll
      for (int t = 0; t < 8; ++t) mv[t] = fmaxf(mv[t], fabsf(x[t]));
    }
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
  for (int t = 0; t < 8; ++t) vcol[hw][col + t] = mv[t];
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f, b = 0.f;
    for (int w = 0; w < kWarps; ++w) {
      a = fmaxf(a, red[0][w]);
      b = fmaxf(b, red[1][w]);
    }
    atomicMax(amax + bh, __float_as_uint(a));
    if (has_kv) atomicMax(amax + BH + bh, __float_as_uint(b));
  }
  if (!has_kv || threadIdx.x >= D) return;
  const int c = threadIdx.x;  // one column per thread
  float m = 0.f;
  for (int h = 0; h < 2 * kWarps; ++h) m = fmaxf(m, vcol[h][c]);
  atomicMax(amax + BH + BHkv + static_cast<size_t>(bh) * D + c, __float_as_uint(m));
}

__global__ void __launch_bounds__(kQuantThreads)
    fp8_quant_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                     const __nv_bfloat16* __restrict__ v, const float* __restrict__ signs, int BH,
                     int BHkv, int N, int Np, const unsigned int* __restrict__ amax,
                     uint8_t* __restrict__ q8, uint8_t* __restrict__ k8, uint8_t* __restrict__ vt8) {
  constexpr int D = 128;
  constexpr int kWarps = kQuantThreads / 32;
  const int bh = blockIdx.y, blk = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = 2 * warp + (lane >> 4), col = 8 * (lane & 15);
  __shared__ __align__(16) uint32_t vt[D * kTile / 4];  // V^T of the block, swizzled words
  const bool rot = signs != nullptr;
  const bool has_kv = bh < BHkv;
  const float iq = 1.f / scale_of(__uint_as_float(amax[bh]));
  const float ik = has_kv ? 1.f / scale_of(__uint_as_float(amax[BH + bh])) : 1.f;
  constexpr float kInvSqrt = 0.08838834764831845f;  // 1 / sqrt(128)
  float fq[8], fk[8], iv[8];  // per column: sign / sqrt(128) / scale (Q, K); 1 / scale (V)
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const float g = rot ? signs[col + t] * kInvSqrt : 1.f;
    fq[t] = g * iq;
    fk[t] = g * ik;
    iv[t] = has_kv ? 1.f / scale_of(__uint_as_float(
                               amax[BH + BHkv + static_cast<size_t>(bh) * D + col + t]))
                   : 1.f;
  }
  const int rows = min(kTile, N - blk * kTile);
  for (int r0 = 0; r0 < kTile; r0 += kQuantRowsPerIter) {
    uint4 wq[2], wk[2], wv[2];
    bool in[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int rr = r0 + hw + u * (2 * kWarps);
      in[u] = rr < rows;
      const size_t off = (static_cast<size_t>(bh) * N + blk * kTile + rr) * D + col;
      wq[u] = in[u] ? load8(q + off) : make_uint4(0, 0, 0, 0);
      wk[u] = in[u] && has_kv ? load8(k + off) : make_uint4(0, 0, 0, 0);
      wv[u] = in[u] && has_kv ? load8(v + off) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int rr = r0 + hw + u * (2 * kWarps);
      const size_t off = (static_cast<size_t>(bh) * N + blk * kTile + rr) * D + col;
      float x[8];
      unpack8(wq[u], x);
      if (rot) {
        hadamard128(x, fq);  // every lane of the warp takes part in the shuffles
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] *= iq;
      }
      if (in[u]) *reinterpret_cast<uint2*>(q8 + off) = e4m3x8(x);
      unpack8(wk[u], x);
      if (rot) {
        hadamard128(x, fk);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t) x[t] *= ik;
      }
      if (in[u] && has_kv) *reinterpret_cast<uint2*>(k8 + off) = e4m3x8(x);
      unpack8(wv[u], x);
#pragma unroll
      for (int t = 0; t < 8; ++t) x[t] *= iv[t];
      const uint2 cv = e4m3x8(x);  // rows past N hold zero codes: V^T's padding
      uint8_t* vtb = reinterpret_cast<uint8_t*>(vt);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int c = col + t;
        vtb[4 * (c * (kTile / 4) + ((rr >> 2) ^ vt_swz(c))) + (rr & 3)] =
            static_cast<uint8_t>((t < 4 ? cv.x : cv.y) >> (8 * (t & 3)));
      }
    }
  }
  __syncthreads();
  if (!has_kv) return;
  // V^T rows of this block: column c, keys blk*128 .. blk*128 + 127 (zeros past N),
  // written 16 bytes at a time up to the padded length Np.
  for (int i = threadIdx.x; i < D * (kTile / 16); i += kQuantThreads) {
    const int c = i / (kTile / 16), seg = i % (kTile / 16);
    const int key0 = blk * kTile + seg * 16;
    if (key0 >= Np) continue;
    const uint32_t* col_words = vt + c * (kTile / 4);
    const int z = vt_swz(c);
    const uint4 w = make_uint4(col_words[(4 * seg) ^ z], col_words[(4 * seg + 1) ^ z],
                               col_words[(4 * seg + 2) ^ z], col_words[(4 * seg + 3) ^ z]);
    *reinterpret_cast<uint4*>(vt8 + (static_cast<size_t>(bh) * D + c) * Np + key0) = w;
  }
}

__global__ void fp8_scales_kernel(const unsigned int* __restrict__ amax, int BH, int BHkv,
                                  float* __restrict__ s_q, float* __restrict__ s_k,
                                  float* __restrict__ s_v) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < BH) s_q[i] = scale_of(__uint_as_float(amax[i]));
  if (i < BHkv) s_k[i] = scale_of(__uint_as_float(amax[BH + i]));
  if (i < BHkv * 128) s_v[i] = scale_of(__uint_as_float(amax[BH + BHkv + i]));
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, cudaStream_t stream) {
  const int BH = a.B * a.H, BHkv = a.B * a.Hkv;  // Hkv divides H, so BHkv <= BH
  const dim3 grid((a.N + kTile - 1) / kTile, BH);
  cudaError_t e = cudaMemsetAsync(
      a.amax, 0, sizeof(unsigned int) * (static_cast<size_t>(BH) + 129 * static_cast<size_t>(BHkv)),
      stream);
  if (e != cudaSuccess) return e;
  fp8_amax_kernel<<<grid, kQuantThreads, 0, stream>>>(a.q, a.k, a.v, a.signs, BH, BHkv, a.N,
                                                      a.amax);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_quant_kernel<<<grid, kQuantThreads, 0, stream>>>(a.q, a.k, a.v, a.signs, BH, BHkv, a.N,
                                                       a.Np, a.amax, a.q8, a.k8, a.vt8);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  fp8_scales_kernel<<<(BH * 128 + 255) / 256, 256, 0, stream>>>(a.amax, BH, BHkv, a.s_q, a.s_k,
                                                                a.s_v);
  return cudaGetLastError();
}

}  // namespace fa
