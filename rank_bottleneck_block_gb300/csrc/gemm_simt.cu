// fp32 SIMT GEMM instantiations (one per epilogue).
#include "simt_gemm.cuh"

namespace lr {
#define LR_INST(K, NACC) template cudaError_t launch_simt<K, NACC>(const GemmCall&, cudaStream_t);
LR_INST(EPI_NORM_SILU, 1)
LR_INST(EPI_SILU, 1)
LR_INST(EPI_STORE, 1)
LR_INST(EPI_RESID, 1)
LR_INST(EPI_SWIGLU, 2)
LR_INST(EPI_DSILU, 1)
LR_INST(EPI_DSILU_NORM, 1)
LR_INST(EPI_SWIGLU_BWD, 1)
LR_INST(EPI_DX_NORM, 1)
LR_INST(EPI_F32, 1)
#undef LR_INST
}  // namespace lr
