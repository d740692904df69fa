// tcgen05 GEMM instantiations of the forward epilogues (operands K-major).
#include "umma_launch.cuh"

namespace lr {
#define LR_INST(K, BN, AMN, BMN) \
  template cudaError_t launch_umma<K, BN, AMN, BMN>(const GemmCall&, cudaStream_t);
LR_INST(EPI_NORM_SILU, 128, false, false)
LR_INST(EPI_NORM_SILU, 256, false, false)
LR_INST(EPI_SILU, 128, false, false)
LR_INST(EPI_SILU, 256, false, false)
LR_INST(EPI_STORE, 128, false, false)
LR_INST(EPI_STORE, 256, false, false)
LR_INST(EPI_RESID, 128, false, false)
LR_INST(EPI_RESID, 256, false, false)
LR_INST(EPI_SWIGLU, 128, false, false)
LR_INST(EPI_SWIGLU, 256, false, false)
LR_INST(EPI_NORM_SWIGLU, 256, false, false)
LR_INST(EPI_SWIGLU_H, 256, false, false)
LR_INST(EPI_F32_SS, 128, false, false)
LR_INST(EPI_F32_SS, 256, false, false)
#undef LR_INST
}  // namespace lr
