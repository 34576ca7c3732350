// Internal interface between the C-ABI layer (fa_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

struct FwdArgs {
  MaskParams mask;
  DropParams drop;
  SyncParams sync;
  float scale_log2;  // scale * log2(e)
  __nv_bfloat16* o;  // [B, H, N, d]
  float* lse;        // [B, H, N]
};

struct BwdArgs {
  MaskParams mask;
  DropParams drop;
  SyncParams sync;
  float scale;       // softmax scale (dK and dQ are multiplied by it)
  float scale_log2;  // scale * log2(e)
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;  // [B, H, N], natural log
  float* dsum;       // D = rowsum(dO * O), fp32 [B, H, N] (workspace)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
};

// Short-query attention over a K/V cache (fa_decode.cu). The work is the
// flattened list of (K/V head, key tile) pairs, B * Hkv * n_t long; CTA c
// takes the pairs [c * per_cta, (c + 1) * per_cta). A K/V head that falls into
// one CTA's range is finished there (O, lse written directly); a head cut by
// CTA boundaries leaves one normalised partial result per piece, merged by
// the combine kernel.
struct DecodeArgs {
  int B, H, Hkv, Nq, Nk;        // query heads H share Hkv K/V heads; Nq query rows, Nk cache rows
  int causal;                   // query row i sits at position L_b - Nq + i
  int wl;                       // sliding window: keys >= L_b - Nq + i - wl only (-1: none)
  const int32_t* seqlens_k;     // [B] valid cache lengths L_b, or null (= Nk)
  int n_t;                      // ceil(Nk / 128): key tiles per K/V head
  int per_cta;                  // (K/V head, key tile) pairs per CTA
  int seg_max;                  // partial-result slots per query row
  float scale_log2;             // scale * log2(e)
  SyncParams sync;
  __nv_bfloat16* o;             // [B, H, Nq, d]
  float* lse;                   // [B, H, Nq]
  float* o_part;                // [B*H*Nq, seg_max, d] fp32 (heads cut by CTA boundaries)
  float* lse_part;              // [B*H*Nq, seg_max]
};

cudaError_t launch_decode(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeArgs& a, int d, int grid, cudaStream_t stream);
cudaError_t launch_decode_combine(const DecodeArgs& a, int d, cudaStream_t stream);

// FP8 forward (fa_fp8.cu, fa_fwd_fp8.cu), head dimension 128.
struct Fp8QuantArgs {
  const __nv_bfloat16* q;          // [B, H, N, 128]
  const __nv_bfloat16 *k, *v;      // [B, Hkv, N, 128]
  const float* signs;              // [128], +-1: the rotation's random signs
  int B, H, Hkv, N, Np;            // Np: row stride of vt8, N rounded up to 16
  unsigned int* amax;              // workspace [B*H + 129*B*Hkv]
  uint8_t* q8;                     // e4m3 [B, H, N, 128] (rotated, scaled)
  uint8_t* k8;                     // e4m3 [B, Hkv, N, 128] (rotated, scaled)
  uint8_t* vt8;                    // e4m3 [B, Hkv, 128, Np] (V transposed, scaled per column)
  float* s_q;                      // [B*H]
  float* s_k;                      // [B*Hkv]
  float* s_v;                      // [B*Hkv, 128]
};

struct Fp8FwdArgs {
  MaskParams mask;
  SyncParams sync;
  float scale_log2;                // softmax scale * log2(e)
  const float *s_q, *s_k, *s_v;
  __nv_bfloat16* o;                // [B, H, N, 128]
  float* lse;                      // [B, H, N]
};

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, cudaStream_t stream);
cudaError_t launch_fwd_fp8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                           const Fp8FwdArgs& a, int num_sms, cudaStream_t stream);

// Tensor maps of a [B*H, N, d] bf16 tensor with 128 x 64 boxes, 128-byte swizzle.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool dropout, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(const BwdArgs& a, int d, int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_dkdv(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdArgs& a, int d, bool dropout,
                            int num_sms, cudaStream_t stream);

cudaError_t launch_bwd_dq(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdArgs& a, int d, bool dropout,
                          int num_sms, cudaStream_t stream);

// Two-issuer backward kernels (fa_bwd_split.cu): dK/dV at d = 64 (d = 128 runs the
// single-issuer kernel of fa_bwd.cu), dQ at d = 64 or 128.
cudaError_t launch_bwd_dkdv_split(const CUtensorMap& tq, const CUtensorMap& tk,
                                  const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                                  int d, bool dropout, int num_sms, cudaStream_t stream);
cudaError_t launch_bwd_dq_split(const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const CUtensorMap& tdo, const BwdArgs& a,
                                int d, bool dropout, int num_sms, cudaStream_t stream);

cudaError_t launch_debug_dropout(uint8_t* keep, int B, int H, int N, const DropParams& d,
                                 cudaStream_t stream);

cudaError_t launch_debug_philox(const uint32_t* counters, uint32_t* out, int n, uint32_t k0,
                                uint32_t k1, cudaStream_t stream);

}  // namespace fa
