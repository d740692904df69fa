// Host launcher of the tcgen05 GEMM: builds the TMA tensor maps of the
// operands, of the epilogue's operand tiles and of its outputs, and starts a
// persistent grid of at most one CTA per SM.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
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

// Tiled map over a row-major array: dims[0] is the contiguous dimension; strides in elements.
inline bool encode(CUtensorMap* m, CUtensorMapDataType dt, int esize, const void* ptr, int rank,
                   const long long* dims, const long long* strides, const int* box, CUtensorMapSwizzle swz) {
  auto fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t gd[3], gs[2];
  cuuint32_t bx[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gd[i] = static_cast<cuuint64_t>(dims[i]);
    bx[i] = static_cast<cuuint32_t>(box[i]);
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = static_cast<cuuint64_t>(strides[i]) * esize;
  CUresult r = fn(m, dt, rank, const_cast<void*>(ptr), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [outer, inner] with row pitch ld: mainloop operand tiles, 128-byte swizzle.
inline bool encode_operand(CUtensorMap* m, const void* ptr, long long inner, long long outer, long long ld,
                           int box_inner, int box_outer) {
  const long long dims[2] = {inner, outer}, strides[1] = {ld};
  const int box[2] = {box_inner, box_outer};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// bf16 [M, N] epilogue tile map (32 columns x 32 rows: one warp's rows, 64-byte swizzle).
inline bool encode_epi_bf16(CUtensorMap* m, const void* ptr, long long N, long long M, long long ld) {
  const long long dims[2] = {N, M}, strides[1] = {ld};
  const int box[2] = {CW, ER};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

// fp32 [splits, M, N] partial-output map (32 columns x 32 rows x 1 split, 128-byte swizzle).
inline bool encode_epi_f32(CUtensorMap* m, const void* ptr, long long N, long long M, long long ld, long long splits,
                           long long split_stride) {
  const long long dims[3] = {N, M, splits}, strides[2] = {ld, split_stride};
  const int box[3] = {CW, ER, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, ptr, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace umma

template <EpiKind K, int BN, bool A_MN, bool B_MN, bool RB>
cudaError_t launch_umma(const GemmCall& g, cudaStream_t st) {
  using namespace umma;
  using C = Config<K, BN>;
  using D = EpiDef<K>;
  constexpr int NACC = D::NACC;
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  Shape sh;
  memset(&sh, 0, sizeof(sh));
  sh.M = g.M;
  sh.N = g.N;
  sh.K = g.K;
  sh.batches = NACC > 1 && !g.rowbatch ? 1 : g.batches;
  sh.m_tiles = (g.M + BM - 1) / BM;
  sh.n_tiles = (g.N + BN - 1) / BN;
  sh.m_pairs = (sh.m_tiles + 1) / 2;
  sh.kb_total = (g.K + BK - 1) / BK;
  const int ks = g.ksplit < 1 ? 1 : g.ksplit;
  sh.kb_per_split = (sh.kb_total + ks - 1) / ks;
  sh.ksplit = (sh.kb_total + sh.kb_per_split - 1) / sh.kb_per_split;  // no empty split
  sh.err = g.err;
  sh.reverse = g.reverse ? 1 : 0;
  if (g.rowbatch != RB) return cudaErrorInvalidValue;
  if (!g.rowbatch && !g.grouped && NACC == 1 && (g.batches < 1 || g.batches > kMaxBatch)) return cudaErrorInvalidValue;
  if (g.rowbatch) {  // one tensor per operand, batches offset by rows
    if (D::NAUX > 0 || C::STATS || ((C::SPLIT || NACC > 1) && K != EPI_ATTN_BWD) || D::ROWPART || g.grouped ||
        sh.ksplit != 1 || g.M % (2 * BM) || g.N % BN || g.K % BK || g.bh < 0 ||
        g.rb_a < 0 || g.rb_b < 0 || g.rb_o < 0 || g.rl_a < 0 || g.rl_b < 0 || g.rl_o < 0 ||
        g.cb_a < 0 || g.cb_b < 0 || g.cb_o < 0 || g.cb_a % 8 || g.cb_b % 8 || g.cb_o % 8 ||
        g.cols_a < 0 || g.cols_b < 0 || g.cols_o < 0)
      return cudaErrorInvalidValue;
    sh.rowbatch = 1;
    sh.bh = g.bh > 0 ? g.bh : 1;
    sh.rb_a = g.rb_a;
    sh.rb_b = g.rb_b;
    sh.rb_o = g.rb_o;
    sh.rl_a = g.rl_a;
    sh.rl_b = g.rl_b;
    sh.rl_o = g.rl_o;
    sh.cb_a = g.cb_a;
    sh.cb_b = g.cb_b;
    sh.cb_o = g.cb_o;
    sh.causal = g.causal;
  }
  if (g.causal && (!g.rowbatch || g.causal > 3 || g.M % (2 * BM) || (g.causal == 1 && g.N != g.M)))
    return cudaErrorInvalidValue;
  sh.grouped = 0;
  if (g.grouped) {  // batches of their own M, N; one split only
    if (K != EPI_F32 || sh.ksplit != 1 || g.batches < 1 || g.batches > kMaxBatch) return cudaErrorInvalidValue;
    sh.grouped = 1;
    int t = 0;
    for (int b = 0; b < kMaxBatch; ++b) {
      sh.g_n_tiles[b] = b < g.batches ? (g.gN[b] + BN - 1) / BN : 1;
      sh.g_tile0[b] = t;
      if (b < g.batches) t += ((g.gM[b] + 2 * BM - 1) / (2 * BM)) * sh.g_n_tiles[b];
    }
    sh.g_tiles = t;
  }
  // Extent of batch (or operand set) b.
  auto bM = [&](int b) { return g.grouped ? g.gM[b] : g.M; };
  auto bN = [&](int b) { return g.grouped ? g.gN[b] : g.N; };
  // Stored rows of operand A / B / the output (all batches' rows when row-batched).
  auto rowsA = [&](int b) -> long long { return g.rowbatch ? g.rows_a : (A_MN ? g.K : bM(b)); };
  // B of operand set b MN-major: the kernel's B_MN, or a set the kind reads MN-major
  auto bmn = [&](int b) { return B_MN || ((C::B_MN_SETS >> b) & 1u); };
  auto rowsB = [&](int b) -> long long { return g.rowbatch ? g.rows_b : (bmn(b) ? g.K : bN(b)); };
  // Stored columns (the inner extent): all batches' columns when row-batched with column offsets.
  auto colsA = [&](int b) -> long long { return g.rowbatch && g.cols_a ? g.cols_a : (A_MN ? bM(b) : g.K); };
  auto colsB = [&](int b) -> long long { return g.rowbatch && g.cols_b ? g.cols_b : (bmn(b) ? bN(b) : g.K); };

  const int nsets = NACC > 1 ? NACC : (g.rowbatch ? 1 : g.batches);
  for (int i = 0; i < nsets; ++i) {
    const bool okA = A_MN ? encode_operand(&maps.a[i], g.A[i].ptr, colsA(i), rowsA(i), g.A[i].ld, 64, 64)
                          : encode_operand(&maps.a[i], g.A[i].ptr, colsA(i), rowsA(i), g.A[i].ld, 64, BM);
    // Each CTA of a pair stages half of the B tile: BN/2 rows (K-major) or 64-column chunks (MN-major).
    const bool okB = bmn(i) ? encode_operand(&maps.b[i], g.B[i].ptr, colsB(i), rowsB(i), g.B[i].ld, 64, 64)
                          : encode_operand(&maps.b[i], g.B[i].ptr, colsB(i), rowsB(i), g.B[i].ld, 64, BN / 2);
    if (!okA || !okB) return cudaErrorInvalidValue;
  }
  const void* const* outs[3] = {g.ep.out0, g.ep.out1, g.ep.out2};
  const long long ldo[3] = {g.ep.ldo0, g.ep.ldo1, g.ep.ldo2};
  const void* const* auxs[2] = {g.ep.aux0, g.ep.aux1};
  const long long lda[2] = {g.ep.lda0, g.ep.lda1};
  const int nmaps = g.rowbatch ? 1 : sh.batches;
  for (int b = 0; b < nmaps; ++b) {
    for (int o = 0; o < D::NOUT; ++o) {
      const void* p = outs[o][b];
      if (!p) continue;
      const long long ld = g.grouped ? g.gldo[b] : ldo[o];
      const long long orows = g.rowbatch ? g.rows_o : bM(b);
      const long long ocols = g.rowbatch && g.cols_o ? g.cols_o : bN(b);
      const long long stride = g.grouped ? ld * bM(b) : (g.rowbatch ? ld * orows : g.ep.split_stride);
      const bool ok = D::OUT_F32 ? encode_epi_f32(&maps.out[b][o], p, ocols, orows, ld, sh.ksplit, stride)
                                 : encode_epi_bf16(&maps.out[b][o], p, ocols, orows, ld);
      if (!ok) return cudaErrorInvalidValue;
    }
    for (int a = 0; a < D::NAUX; ++a) {
      const void* p = auxs[a][b];
      if (!p) continue;
      if (!encode_epi_bf16(&maps.aux[b][a], p, g.N, g.M, lda[a])) return cudaErrorInvalidValue;
    }
  }

  const long long total =  // pair tiles
      1LL * sh.ksplit * (sh.grouped ? sh.g_tiles : sh.batches * batch_tiles<RB>(sh));
  if (total <= 0) return cudaSuccess;

  auto kern = gemm_kernel<K, BN, A_MN, B_MN, RB>;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;  // a CTA pair on two SMs
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;

  // Per device, once: the shared-memory opt-in and how many pairs can be resident at once.
  static int configured_mask = 0;
  static int max_pairs[32];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 32) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // The kernel's setmaxnreg split must fit the registers it is launched with (a split above
    // them would leave the epilogue warps waiting for registers forever): checked once here.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    if (C::REGSPLIT && 1LL * fa.numRegs * C::THREADS < 128LL * kRegCtl + 256LL * kRegEpi)
      return cudaErrorInvalidConfiguration;
    cfg.gridDim = dim3(2, 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = device_sm_count() / 2;
    }
    max_pairs[dev] = n;
    __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  // The fewest pairs that take the tiles in the same number of waves: the makespan of the static
  // round-robin schedule is unchanged and the SMs left over stay free for concurrent work (a second
  // stream's kernels; the next kernel's prologue).  Causal launches, whose tiles differ in length,
  // keep every pair.
  long long pairs = total < max_pairs[dev] ? total : max_pairs[dev];
  if (g.max_pairs > 0 && pairs > g.max_pairs) pairs = g.max_pairs;
  if (g.causal == 0 && pairs > 0) {
    const long long waves = (total + pairs - 1) / pairs;
    pairs = (total + waves - 1) / waves;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs), 1, 1);
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, maps, sh, g.ep);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace lr
