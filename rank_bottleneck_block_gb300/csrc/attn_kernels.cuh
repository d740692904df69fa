// Row kernels of causal multi-head attention between the low-rank projections (bf16
// storage, fp32 arithmetic): the forward softmax and the backward's row dot D = rowsum(dO * O).
// The GEMMs run on the tcgen05 engine in row-batched mode over all heads (the backward's P and
// dS come out of one dual-accumulator GEMM's epilogue).  Score rows are head-major: row
// r = (bi*H + h)*s + i is query i of head h of sequence bi.  q, k, v, o and dO are token-major
// ([b*s, H*dh], head h of token t in columns h*dh .. h*dh + dh - 1).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace lr {

// Row r of S [R, s] fp32 (R = heads * s; query i = r mod s; only j <= i is read) -> P [R, s] bf16
// with P_rj = exp(scale S_rj - lse_r) for j <= i and 0 for i < j < the end of i's 256-row tile
// (columns past it are not written), and lse_r = log sum_{j<=i} exp(scale S_rj).
cudaError_t launch_attn_softmax_fwd(const float* S, int R, int s, float scale, bf16* P, float* lse,
                                    cudaStream_t st);

// D_r = sum_c dO[t, h*dh + c] O[t, h*dh + c] for score row r (query i of head h of sequence bi,
// token t = bi*s + i), over the dh columns of the head.  dh a multiple of 8.
cudaError_t launch_attn_rowdot(const bf16* dO, const bf16* O, int b, int s, int H, int dh, float* D,
                               cudaStream_t st);

// Causal attention forward without materialised scores (tcgen05; the head width it is built for):
// o [b*s, H*dh] token-major and lse [b*H*s] head-major (natural log), from token-major q, k, v.  s a
// multiple of 128; every wait bounded (a timeout sets a bit of *err).  sched: one device word, the
// launch's work-item counter (cleared on `st` before the launch; no other use may overlap the launch).
bool attn_flash_fwd_supported(int dh);
cudaError_t launch_attn_flash_fwd(const bf16* q, const bf16* k, const bf16* v, bf16* o, int b, int s, int H, int dh,
                                  float scale, float* lse, unsigned* sched, unsigned* err, cudaStream_t st);

// Causal attention backward without materialised P (tcgen05; the head width it is built for): dk, dv
// [b*s, H*dh] token-major and dst = scale dS^T, head-major [b*H*s keys, s queries] bf16 (the blocks on
// and below the diagonal, plus key block j against query block j - 1 for odd j, zero), from token-major
// q, k, v, dout, the forward's lse and D_q = sum_c dO_qc O_qc (both head-major [b*H*s]).  s a multiple of
// 128; sched as for the forward.
cudaError_t launch_attn_flash_bwd(const bf16* q, const bf16* k, const bf16* v, const bf16* dout, const float* lse,
                                  const float* D, bf16* dst, bf16* dk, bf16* dv, int b, int s, int H, int dh,
                                  float scale, unsigned* sched, unsigned* err, cudaStream_t st);

}  // namespace lr
