// tcgen05 GEMM instantiations of the backward epilogues (B operand MN-major:
// dX = dY . W reads W in its stored orientation; weight gradients read both
// operands MN-major, K = tokens).
#include "umma_launch.cuh"

namespace lr {
#define LR_INST(K, BN, NACC, AMN, BMN) \
  template cudaError_t launch_umma<K, BN, NACC, AMN, BMN>(const GemmCall&, cudaStream_t);
LR_INST(EPI_DSILU, 128, 1, false, true)
LR_INST(EPI_DSILU, 256, 1, false, true)
LR_INST(EPI_DSILU_NORM, 128, 1, false, true)
LR_INST(EPI_DSILU_NORM, 256, 1, false, true)
LR_INST(EPI_SWIGLU_BWD, 128, 1, false, true)
LR_INST(EPI_SWIGLU_BWD, 256, 1, false, true)
LR_INST(EPI_DX_NORM, 128, 1, false, true)
LR_INST(EPI_DX_NORM, 256, 1, false, true)
LR_INST(EPI_STORE, 128, 1, false, true)
LR_INST(EPI_STORE, 256, 1, false, true)
LR_INST(EPI_F32, 128, 1, true, true)
LR_INST(EPI_F32, 256, 1, true, true)
#undef LR_INST
}  // namespace lr
