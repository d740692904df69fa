// Row kernels of causal multi-head attention between the low-rank projections (bf16
// storage, fp32 arithmetic).  The GEMMs run on the tcgen05 engine in row-batched mode over
// head-major tensors (the backward's P and dS come out of one dual-accumulator GEMM's
// epilogue); these kernels move heads between the token-major layout the projections use
// ([b*s, H*dh], head h of token t in columns h*dh .. h*dh + dh - 1) and the head-major one
// ([b*H*s, dh], head (bi, h) in rows (bi*H + h)*s .. + s - 1), and do the forward softmax
// and the backward's row dot D = rowsum(dO * O).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace lr {

// to_heads != 0: dst (head-major) <- src (token-major); else dst (token-major) <- src (head-major).
// dh a multiple of 8.
cudaError_t launch_head_permute(const bf16* src, bf16* dst, int b, int s, int H, int dh, int to_heads,
                                cudaStream_t st);

// Row r of S [R, s] fp32 (R = heads * s; query i = r mod s; only j <= i is read) -> P [R, s] bf16
// with P_rj = exp(scale S_rj - lse_r) for j <= i and 0 for i < j < the end of i's 256-row tile
// (columns past it are not written), and lse_r = log sum_{j<=i} exp(scale S_rj).
cudaError_t launch_attn_softmax_fwd(const float* S, int R, int s, float scale, bf16* P, float* lse,
                                    cudaStream_t st);

// D_r = sum_c dO[r, c] O[r, c] over the dh columns of head-major rows.
cudaError_t launch_attn_rowdot(const bf16* dO, const bf16* O, int R, int dh, float* D, cudaStream_t st);

}  // namespace lr
