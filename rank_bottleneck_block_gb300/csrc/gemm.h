// Host-side description of one fused GEMM launch and the launchers of the two
// GEMM engines: the tcgen05 kernel (bf16 operands) and the SIMT kernel (fp32
// operands, exact fp32 arithmetic, no TF32).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace lr {

// A matrix operand stored row-major with leading dimension `ld` (elements).
// For operand A ([M, K] logically): K-major storage holds element (m, k) at
// ptr[m * ld + k]; MN-major storage holds it at ptr[k * ld + m].
// Operand B ([N, K] logically) is read the same way with n in place of m.
struct Operand {
  const void* ptr;
  long long ld;
};

struct GemmCall {
  int M, N, K;
  int nacc;     // accumulators per tile (2: SwiGLU dual GEMM, segment s uses A[s], B[s])
  int batches;  // independent problems of the same shape (batch b uses A[b], B[b])
  int ksplit;   // split-K factor (EPI_F32 only): partial s goes to out0 + s * split_stride
  bool a_mn, b_mn;
  Operand A[kMaxBatch];
  Operand B[kMaxBatch];
  EpiParams ep;
  unsigned* err;  // device error word
  int bn;         // tcgen05 tile width chosen by the planner (128 or 256)
  // Walk the tiles from the last one: a GEMM that reads a large tensor the previous kernel
  // wrote in tile order then starts on its most recently written (still L2-resident) part.
  bool reverse;
  // Grouped problems (EPI_F32, tcgen05 path, no split): batch b has its own gM[b] x gN[b] output
  // with leading dimension gldo[b] (elements); all batches share K, the tile width and the operand
  // layouts, and their tiles are scheduled as one persistent grid.  False: uniform batches of M x N.
  bool grouped;
  int gM[kMaxBatch], gN[kMaxBatch];
  long long gldo[kMaxBatch];
  // Row-batched problems (kinds without operand tiles, row statistics or row partials): every
  // batch reads and writes one tensor per operand at an offset, so any number of batches shares
  // one set of tensor maps.  Batch b = hi bh + lo (bh >= 1) of operand X starts hi rb_X + lo rl_X
  // stored rows and lo cb_X stored columns in (rows_X stored rows in all; cols_X stored columns,
  // or 0 for the batch's own extent).  A stored row is an M index for a K-major A and a K index
  // for an MN-major one (likewise N or K for B), a stored column the other index.  Each batch's
  // M, N and K must be whole tiles: M a multiple of 256, N of the tile width, K of 64; column
  // offsets multiples of 8.
  bool rowbatch;
  int bh;
  int rb_a, rb_b, rb_o, rl_a, rl_b, rl_o, cb_a, cb_b, cb_o;
  long long rows_a, rows_b, rows_o, cols_a, cols_b, cols_o;
  // Causal masking of a row-batched attention GEMM over s positions (rows and columns or K index
  // positions, whole pair tiles of 256): 1 = rows are queries and columns keys (M = N), only the
  // tiles on or below the diagonal are scheduled; 2 = rows are queries and K keys, K stops after the tile's last row;
  // 3 = rows are keys and K queries, K starts at the tile's first row.  0: none.
  int causal;
  // At most this many SM pairs (0: as many as the tiles can use); the rest stay free for a kernel on
  // another stream.
  int max_pairs;
};

// Row-partial chunk width used by the epilogues of each engine.
constexpr int kChunkUmma = 32;  // the tcgen05 epilogue chunk (umma::CW)
constexpr int kChunkSimt = 8;

// RB: the kernel built for row-batched calls (g.rowbatch must equal it).
template <EpiKind K, int BN, bool A_MN, bool B_MN, bool RB = false>
cudaError_t launch_umma(const GemmCall& g, cudaStream_t st);

template <EpiKind K>
cudaError_t launch_simt(const GemmCall& g, cudaStream_t st);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace lr
