// tcgen05 GEMM instantiations built for row-batched calls: causal attention over all heads.
// S = Q K^T with fp32 output (both operands K-major), O = P V and dQ = dS K (B MN-major),
// dK = dS^T Q and dV = P^T dO (both MN-major), and the backward's dual-accumulator scores
// kernel (S = Q K^T and dP = dO V^T of one tile, out P and dS).
#include "umma_launch.cuh"

namespace lr {
#define LR_INST(K, BN, AMN, BMN) \
  template cudaError_t launch_umma<K, BN, AMN, BMN, true>(const GemmCall&, cudaStream_t);
LR_INST(EPI_F32, 128, false, false)
LR_INST(EPI_F32, 256, false, false)
LR_INST(EPI_STORE, 128, false, true)
LR_INST(EPI_STORE, 256, false, true)
LR_INST(EPI_STORE, 128, true, true)
LR_INST(EPI_STORE, 256, true, true)
LR_INST(EPI_ATTN_BWD, 256, false, false)
#undef LR_INST
}  // namespace lr
