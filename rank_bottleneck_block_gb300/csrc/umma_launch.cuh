// Host launcher of the tcgen05 GEMM: builds the TMA tensor maps of each
// operand and starts a persistent grid of at most one CTA per SM.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "gemm.h"
#include "umma_gemm.cuh"

namespace lr {
namespace umma {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 map over a row-major [outer, inner] array with row pitch ld elements, 128-byte swizzle.
inline bool encode(CUtensorMap* m, const void* ptr, long long inner, long long outer, long long ld, int box_inner,
                   int box_outer) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_outer)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace umma

template <EpiKind K, int BN, int NACC, bool A_MN, bool B_MN>
cudaError_t launch_umma(const GemmCall& g, cudaStream_t st) {
  using namespace umma;
  using C = Config<BN, NACC>;
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  const int nsets = NACC > 1 ? NACC : g.batches;
  for (int i = 0; i < nsets; ++i) {
    const bool okA = A_MN ? encode(&maps.a[i], g.A[i].ptr, g.M, g.K, g.A[i].ld, 64, 64)
                          : encode(&maps.a[i], g.A[i].ptr, g.K, g.M, g.A[i].ld, 64, BM);
    const bool okB = B_MN ? encode(&maps.b[i], g.B[i].ptr, g.N, g.K, g.B[i].ld, 64, 64)
                          : encode(&maps.b[i], g.B[i].ptr, g.K, g.N, g.B[i].ld, 64, BN);
    if (!okA || !okB) return cudaErrorInvalidValue;
  }
  Shape sh;
  sh.M = g.M;
  sh.N = g.N;
  sh.K = g.K;
  sh.batches = NACC > 1 ? 1 : g.batches;
  sh.m_tiles = (g.M + BM - 1) / BM;
  sh.n_tiles = (g.N + BN - 1) / BN;
  sh.kb_total = (g.K + BK - 1) / BK;
  const int ks = g.ksplit < 1 ? 1 : g.ksplit;
  sh.kb_per_split = (sh.kb_total + ks - 1) / ks;
  sh.ksplit = (sh.kb_total + sh.kb_per_split - 1) / sh.kb_per_split;  // no empty split
  sh.err = g.err;
  const long long total = 1LL * sh.ksplit * sh.batches * sh.m_tiles * sh.n_tiles;
  if (total <= 0) return cudaSuccess;
  const int sms = device_sm_count();
  const int grid = static_cast<int>(total < sms ? total : sms);

  auto kern = gemm_kernel<K, BN, NACC, A_MN, B_MN>;
  static int configured_mask = 0;  // one bit per device ordinal
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 31 && !(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  kern<<<grid, kThreads, C::SMEM_BYTES, st>>>(maps, sh, g.ep);
  return cudaGetLastError();
}

}  // namespace lr
