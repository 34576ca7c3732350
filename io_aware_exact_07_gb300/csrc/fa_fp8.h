// Internal interface between the C-ABI layer (fa_api.cu) and the FP8 kernels.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

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

}  // namespace fa
