// fp32 SIMT GEMM with the same fused epilogues as the tcgen05 path.
//
// Serves the fp32 configuration (tensor cores have no exact-fp32 mode and
// TF32 would miss a 1e-5 tolerance).  Each CTA computes a 32 x 64 output tile
// with 256 threads (one row x 8 columns each), staging 16-deep K slices of
// both operands in shared memory; operands may be K-major or MN-major.
#pragma once

#include "epilogues.cuh"
#include "gemm.h"

namespace lr {
namespace simt {

constexpr int TM = 32, TN = 64, TK = 16;

struct Args {
  int M, N, K, batches, ksplit, k_per_split;
  const float* A[kMaxBatch];
  const float* B[kMaxBatch];
  long long a_sm[kMaxBatch], a_sk[kMaxBatch], b_sn[kMaxBatch], b_sk[kMaxBatch];  // per operand set: m / k, n / k
};

template <EpiKind K>
__global__ void __launch_bounds__(256) gemm_kernel(const Args a, const EpiParams ep) {
  pdl_wait();
  pdl_trigger();
  using D = EpiDef<K>;
  constexpr int NACC = D::NACC, NAUX = D::NAUX, NOUT = D::NOUT;
  __shared__ float As[TK][TM + 1];
  __shared__ float Bs[TK][TN + 1];
  const int tid = threadIdx.x;
  const int tr = tid >> 3, tc = tid & 7;
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  const int batch = NACC > 1 ? 0 : static_cast<int>(blockIdx.z) % a.batches;
  const int split = NACC > 1 ? 0 : static_cast<int>(blockIdx.z) / a.batches;
  const int kbeg = split * a.k_per_split;
  const int kend = min(a.K, kbeg + a.k_per_split);
  float acc[NACC][8];
#pragma unroll
  for (int s = 0; s < NACC; ++s)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[s][j] = 0.f;

#pragma unroll
  for (int s = 0; s < NACC; ++s) {
    const int set = NACC > 1 ? s : batch;
    const float* A = a.A[set];
    const float* B = a.B[set];
    for (int k0 = kbeg; k0 < kend; k0 += TK) {
      for (int i = tid; i < TM * TK; i += 256) {
        const int r = i / TK, k = i % TK;
        const int m = m0 + r, kk = k0 + k;
        As[k][r] = (m < a.M && kk < kend) ? A[m * a.a_sm[set] + kk * a.a_sk[set]] : 0.f;
      }
      for (int i = tid; i < TN * TK; i += 256) {
        const int c = i / TK, k = i % TK;
        const int n = n0 + c, kk = k0 + k;
        Bs[k][c] = (n < a.N && kk < kend) ? B[n * a.b_sn[set] + kk * a.b_sk[set]] : 0.f;
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < TK; ++k) {
        const float av = As[k][tr];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[s][j] = fmaf(av, Bs[k][tc * 8 + j], acc[s][j]);
      }
      __syncthreads();
    }
  }
  const int m = m0 + tr, n = n0 + tc * 8;
  if (m >= a.M || n >= a.N) return;
  const RowIn ri = row_inputs<K>(ep, m);
  float av[NAUX > 0 ? NAUX : 1][8];
#pragma unroll
  for (int x = 0; x < NAUX; ++x) {
    const float* p = static_cast<const float*>(epi_aux_ptr(ep, x, batch));
    if (p) {
      load8(p + static_cast<long long>(m) * epi_aux_ld(ep, x) + n, av[x]);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) av[x][j] = 0.f;
    }
  }
  float o[NOUT][8];
  float part = 0.f;
  D::template run<float, 8>(ri, acc, av, o, part);
#pragma unroll
  for (int x = 0; x < NOUT; ++x) {
    float* p = static_cast<float*>(epi_out_ptr(ep, x, batch));
    if (!p) continue;
    if (D::OUT_F32) p += static_cast<long long>(split) * ep.split_stride;
    store8(p + static_cast<long long>(m) * epi_out_ld(ep, x) + n, o[x]);
  }
  if constexpr (D::ROWPART)
    ep.rowpart[(static_cast<long long>(batch) * ep.rowpart_chunks + n / 8) * ep.M + m] = part;
}

}  // namespace simt

template <EpiKind K>
cudaError_t launch_simt(const GemmCall& g, cudaStream_t st) {
  using namespace simt;
  constexpr int NACC = EpiDef<K>::NACC;
  Args a;
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.batches = NACC > 1 ? 1 : g.batches;
  const int ks = g.ksplit < 1 ? 1 : g.ksplit;
  a.k_per_split = ((g.K + ks - 1) / ks + TK - 1) / TK * TK;
  a.ksplit = (g.K + a.k_per_split - 1) / a.k_per_split;
  const int nsets = NACC > 1 ? NACC : g.batches;
  for (int i = 0; i < nsets; ++i) {
    a.A[i] = static_cast<const float*>(g.A[i].ptr);
    a.B[i] = static_cast<const float*>(g.B[i].ptr);
    a.a_sm[i] = g.a_mn ? 1 : g.A[i].ld;
    a.a_sk[i] = g.a_mn ? g.A[i].ld : 1;
    a.b_sn[i] = g.b_mn ? 1 : g.B[i].ld;
    a.b_sk[i] = g.b_mn ? g.B[i].ld : 1;
  }
  dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM, a.batches * a.ksplit);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  return launch_pdl(gemm_kernel<K>, grid, dim3(256), 0, st, a, g.ep);
}

}  // namespace lr
