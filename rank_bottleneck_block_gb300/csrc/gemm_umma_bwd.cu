// tcgen05 GEMM instantiations of the backward epilogues (B operand MN-major:
// dX = dY . W reads W in its stored orientation; weight gradients read both
// operands MN-major, K = tokens).
#include "umma_launch.cuh"

namespace lr {
#define LR_INST(K, BN, AMN, BMN) \
  template cudaError_t launch_umma<K, BN, AMN, BMN>(const GemmCall&, cudaStream_t);
LR_INST(EPI_DSILU, 128, false, true)
LR_INST(EPI_DSILU, 256, false, true)
LR_INST(EPI_DSILU_Z, 128, false, true)
LR_INST(EPI_DSILU_Z, 256, false, true)
LR_INST(EPI_DSILU_NORM, 128, false, true)
LR_INST(EPI_DSILU_NORM, 256, false, true)
LR_INST(EPI_SWIGLU_BWD, 128, false, true)
LR_INST(EPI_SWIGLU_BWD, 256, false, true)
LR_INST(EPI_SWIGLU_BWD_NORM, 128, false, true)
LR_INST(EPI_SWIGLU_BWD_NORM, 256, false, true)
LR_INST(EPI_DX_NORM, 128, false, true)
LR_INST(EPI_DX_NORM, 256, false, true)
LR_INST(EPI_STORE, 128, false, true)
LR_INST(EPI_STORE, 256, false, true)
LR_INST(EPI_F32, 128, true, true)
LR_INST(EPI_F32, 256, true, true)
// the checkpointed re-forward fused with the SwiGLU backward (three K-major accumulators)
LR_INST(EPI_SWIGLU_REBWD, 256, false, false)
#undef LR_INST
}  // namespace lr
