// Internal interface between the C-ABI layer (fa_api.cu) and the bf16 forward and
// backward kernels (and their test hooks); decode and FP8 have their own headers.
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

// Tensor maps of a [B*H, N, d] bf16 tensor with 128 x 64 boxes, 128-byte swizzle.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdArgs& a, int d, bool dropout, int num_sms, cudaStream_t stream);

// d = 128 forward (fa_fwd128.cu); launch_fwd routes d = 128 there.
cudaError_t launch_fwd128(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdArgs& a, bool dropout, int num_sms, cudaStream_t stream);

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
