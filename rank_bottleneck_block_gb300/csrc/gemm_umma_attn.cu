// tcgen05 GEMM instantiations used by causal attention on row-batched heads: S = Q K^T and
// dP = dO V^T with fp32 output (both operands K-major), dK = dS^T Q and dV = P^T dO (both
// operands MN-major).
#include "umma_launch.cuh"

namespace lr {
#define LR_INST(K, BN, AMN, BMN) \
  template cudaError_t launch_umma<K, BN, AMN, BMN>(const GemmCall&, cudaStream_t);
LR_INST(EPI_F32, 128, false, false)
LR_INST(EPI_F32, 256, false, false)
LR_INST(EPI_STORE, 128, true, true)
LR_INST(EPI_STORE, 256, true, true)
#undef LR_INST
}  // namespace lr
