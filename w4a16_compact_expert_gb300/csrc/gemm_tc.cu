// Prefill regime: tensor-core grouped GEMM (tcgen05 / TMEM).  Not built yet.
#include "internal.h"

cudaError_t launch_gemm_experts(const FwdCtx&, cudaStream_t, const StageEvents&) { return cudaErrorNotSupported; }
