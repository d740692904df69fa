// fp32 SIMT GEMM instantiations (one per epilogue).
#include "simt_gemm.cuh"

namespace lr {
#define LR_INST(K) template cudaError_t launch_simt<K>(const GemmCall&, cudaStream_t);
LR_INST(EPI_NORM_SILU)
LR_INST(EPI_SILU)
LR_INST(EPI_STORE)
LR_INST(EPI_RESID)
LR_INST(EPI_SWIGLU)
LR_INST(EPI_DSILU)
LR_INST(EPI_DSILU_NORM)
LR_INST(EPI_SWIGLU_BWD)
LR_INST(EPI_DX_NORM)
LR_INST(EPI_F32)
LR_INST(EPI_NORM_SWIGLU)
LR_INST(EPI_SWIGLU_BWD_NORM)
LR_INST(EPI_F32_SS)
#undef LR_INST
}  // namespace lr
