#include "fa_kernels.h"
namespace fa {
cudaError_t launch_bwd_preprocess(const BwdArgs&, int, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dkdv(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const BwdArgs&, int, bool, int, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_bwd_dq(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, const BwdArgs&, int, bool, int, cudaStream_t) { return cudaErrorNotSupported; }
}
