// Internal interface between the C-ABI layer (fa_api.cu) and the decode kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

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

}  // namespace fa
