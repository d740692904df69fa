// Persistent tcgen05 GEMM for sm_103a with fused, TMA-staged epilogues.
//
//   C[M,N] = sum_k A[m,k] B[n,k]      bf16 operands, fp32 accumulator in TMEM
//
// Mainloop: operands are staged by TMA into a ring of shared-memory stages with
// the 128-byte swizzle; each operand is K-major (rows contiguous in k) or
// MN-major (rows contiguous in m / n: the transposed storage used by the
// weight-gradient and dX = dY . W products), described natively by the UMMA
// shared-memory descriptors, so no transpose kernels exist.
//
// Epilogue: 8 warps in two groups of four; group g handles the 32-column
// chunks c = g, g+2, ... of each tile.  Within a group, warp w reads TMEM lanes
// 32 (w % 4) .. +31 with tcgen05.ld (one output row per thread), the chunk's
// operand tiles (u, a, b, x, dout) arrive by TMA into 64-byte-swizzled shared
// memory, the fused math runs in registers, the results go to swizzled shared
// memory and one thread writes them to global memory with TMA bulk tensor
// stores (rows and columns past the tensor edge are clipped by the TMA unit).
//
// CTA pairs (2-SM UMMA): the kernel runs in clusters of two CTAs on two SMs.
// A pair tile is 256 rows x BN columns; CTA `rank` stages rows 128 rank .. +127
// of A and half of the B tile (BN/2 rows or columns) in its own shared memory,
// and the leader CTA issues tcgen05.mma.cta_group::2 with M = 256, which reads
// both CTAs' operands and leaves rows 128 rank .. +127 of the accumulator in
// each CTA's own TMEM.  Per SM this halves the B-operand traffic through shared
// memory (the mainloop's limit with one CTA per tile) and the B stage size.
//
// Warp roles (320 threads per CTA, one CTA per SM, persistent over pair tiles):
//   warp 0     TMA producer of the CTA's half of the operand ring (one lane)
//   warp 1     TMEM allocator; in the leader CTA also the MMA issuer (one lane)
//   warps 2-3  idle (they complete the first warpgroup, whose registers go to the epilogue)
//   warps 4-11 epilogue of the CTA's 128 rows (two warpgroups)
// setmaxnreg moves registers from the first warpgroup to the epilogue warpgroups.  The kernels
// that compute online-RMSNorm statistics keep the compact layout without the split: warps 2-9
// epilogue, warps 10-13 statistics.
// Two TMEM accumulator buffers let the epilogue of tile i overlap the
// mainloop of tile i+1.  NACC > 1 gives each tile several accumulators fed by
// consecutive K segments with their own operand maps (the SwiGLU dual GEMM).
//
// Every wait on an mbarrier is bounded: after kWaitLimitNs the waiting thread
// sets a bit of the device error word and raises the CTA's abort flag; every
// role then leaves its loop (epilogue groups decide together through a
// barrier reduction), the producer waits (bounded) for its copies in flight,
// the MMA warp drains its issued MMAs, the epilogue waits for its stores, and
// TMEM is freed before the CTA exits.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "epilogues.cuh"

namespace lr {
namespace umma {

constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr int CW = 32;  // epilogue chunk width (columns)
constexpr int ER = 32;  // rows of an epilogue staging tile: one warp's TMEM lane quarter
constexpr int kMaxAuxSets = 4;  // operand-tile staging sets per epilogue warp, at most
constexpr int kMaxAcc = 4;      // TMEM full / empty barrier pairs (a buffer each, or an accumulator each)

// Operand-tile sets per epilogue warp: how many chunks ahead the operand loads run.  The
// residual GEMM (K = r, one [T, d] operand streamed from HBM) gains from four; for the others
// the shared memory is worth more as operand-ring stages (measured: the SwiGLU backward with
// three sets and two stages, and the dz_down GEMM with three sets, were slower).
__host__ __device__ constexpr int aux_sets(EpiKind k) { return k == EPI_RESID ? 4 : 2; }
constexpr int kEpiWarps = 8;
// Register split between the warpgroups (setmaxnreg) of the kernels without statistics warps
// (12 warps): warps 0-3 (producer, MMA issuer / TMEM allocator, two idle warps) keep kRegCtl
// registers per thread, the two epilogue warpgroups take kRegEpi.  The launch gives each thread
// 168 registers (three warps per SM sub-partition); one warp of every warpgroup lives on each
// sub-partition, so the split must satisfy kRegCtl + 2 kRegEpi <= 3 x 168.
constexpr int kRegCtl = 80;
constexpr int kRegEpi = 208;
static_assert(kRegCtl + 2 * kRegEpi <= 3 * 168, "register split of the 12-warp kernels");
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr int kMaxSmem = 227 * 1024;

struct Maps {
  CUtensorMap a[kMaxBatch];
  CUtensorMap b[kMaxBatch];
  CUtensorMap out[kMaxBatch][3];
  CUtensorMap aux[kMaxBatch][2];
};

struct Shape {
  int M, N, K;
  int batches, ksplit;
  int m_tiles, n_tiles;
  int m_pairs;  // pair tiles along M: the CTAs of a cluster take m-tiles 2p and 2p + 1
  int kb_total, kb_per_split;
  int reverse;  // tiles are taken from the last one (see GemmCall::reverse)
  int grouped;  // batches of their own M, N (see GemmCall::grouped); then the next three fields hold
  int g_n_tiles[kMaxBatch];  // n-tiles of batch b
  int g_tile0[kMaxBatch];    // first pair tile of batch b
  int g_tiles;               // pair tiles of all batches
  int rowbatch;              // batches offset into one tensor each (see GemmCall::rowbatch), then
  int bh;                    // batch = hi bh + lo, and A, B, the output start at rows hi rb + lo rl,
  int rb_a, rb_b, rb_o;      //   columns lo cb of their tensors
  int rl_a, rl_b, rl_o;
  int cb_a, cb_b, cb_o;
  int causal;                // causal use of a row-batched problem (see GemmCall::causal), else 0
  unsigned* err;
};

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Returns false (after
// setting `code` in the error word and the CTA abort flag) on timeout or when
// another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* err, unsigned code) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, code);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Shared::cluster address of the same shared variable in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

// A TMA load into this CTA's shared memory whose byte count completes on an mbarrier of
// either CTA of the pair (`bar_cluster` is a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (release at cluster scope).
// Arrive on a barrier of another CTA of the cluster.  Its uses signal that TMEM columns are free:
// the loads that read them have completed (tcgen05.wait::ld, then tcgen05.fence::before_thread_sync)
// and no memory write of the arriving thread is consumed through the barrier, so the release is
// CTA-scoped (the default) rather than cluster-scoped.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// L2 policy that keeps lines in L2 ahead of normal traffic (evict last).
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// tma_store_3d with an L2 cache policy (for data that is read again soon, from L2).
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* map, const void* src, int c0, int c1, int c2,
                                                  uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}

// Explicit 16-byte shared-memory accesses for the staging tiles (their swizzled layout is
// bank-conflict free only when each thread moves whole 16-byte chunks).
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& x, uint32_t& y, uint32_t& z, uint32_t& w) {
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x), "=r"(y), "=r"(z), "=r"(w) : "r"(addr) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& a, float& b) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  a = f.x;
  b = f.y;
}

// Eight bf16 values at a shared address <-> eight floats.
__device__ __forceinline__ void sts_bf16x8(uint32_t addr, const float* v) {
  sts128(addr, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
}

__device__ __forceinline__ void lds_bf16x8(uint32_t addr, float* v) {
  uint32_t w0, w1, w2, w3;
  lds128(addr, w0, w1, w2, w3);
  unpack_bf16x2(w0, v[0], v[1]);
  unpack_bf16x2(w1, v[2], v[3]);
  unpack_bf16x2(w2, v[4], v[5]);
  unpack_bf16x2(w3, v[6], v[7]);
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tmap_prefetch(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Both CTAs of the pair allocate together and receive the same TMEM address.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on the mbarrier at this offset in every CTA of ctamask once the issued MMAs complete.
__device__ __forceinline__ void umma_commit(uint64_t* bar, uint16_t ctamask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(ctamask)
      : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp receives its lane's 32 columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 16 consecutive fp32 columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 at bit 46, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 D, bf16 A and B, operand majors, N >> 3, M >> 4
// (M = 256: the pair's two 128-row halves).
template <int N_, bool A_MN, bool B_MN>
__host__ __device__ constexpr uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N_ >> 3) << 17) | (static_cast<uint32_t>((2 * BM) >> 4) << 24);
}

// Byte offset of 16-byte chunk j of row r in a swizzled staging tile with `row_bytes`
// per row (64: the 64-byte swizzle of bf16 chunks, 128: the 128-byte swizzle of fp32 chunks).
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t stage_off(int r, int j) {
  if constexpr (ROW_BYTES == 64) return r * 64 + ((j ^ ((r >> 1) & 3)) << 4);
  else return r * 128 + ((j ^ (r & 7)) << 4);
}

template <EpiKind K, int BN>
struct Config {
  using D = EpiDef<K>;
  static constexpr int NACC = D::NACC;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = (BN / 2) * BK * 2;  // this CTA's half of the B tile
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int OUT_ROW = CW * (D::OUT_F32 ? 4 : 2);
  static constexpr int OUT_BUF = ER * OUT_ROW;  // one warp's rows of a chunk
  static constexpr int AUX_BUF = ER * CW * 2;
  // The three-accumulator re-forward + SwiGLU backward (a, b, dh of 256 columns each) keeps two
  // TMEM regions of BN columns that its accumulators take in turn: in tile i, a and dh use region
  // i mod 2 (dh once phase 1 has moved a out) and b the other one.
  static constexpr bool TRIPLE = K == EPI_SWIGLU_REBWD;
  static constexpr uint32_t ACC_COLS = TRIPLE ? 2 * BN : NACC * BN;
  // Two accumulator buffers when they fit in the 512 TMEM columns, else one.
  static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;
  // SwiGLU with 256-wide accumulators (a and b fill TMEM): the two accumulators complete and
  // are released separately.  Phase 1 stages round(a) in shared memory (exact: a is stored
  // rounded) and frees a's columns for the next tile while b still accumulates; phase 2 moves
  // round(b) into registers, frees b's columns, then computes h.
  static constexpr bool SPLIT = (K == EPI_SWIGLU || K == EPI_SWIGLU_H || K == EPI_NORM_SWIGLU || K == EPI_ATTN_BWD ||
                                 K == EPI_SWIGLU_REBWD) && NBUF == 1;
  static_assert(!TRIPLE || BN == 256, "the three-accumulator kernel uses two regions of 256 columns");
  // Operand sets whose B is read MN-major whatever the kernel's B_MN: the three-accumulator kernel's
  // dh = du_down A_down reads A_down [r, f] in its stored orientation (sets 0, 1 are K-major).
  static constexpr unsigned B_MN_SETS = TRIPLE ? 4u : 0u;
  // Staging per epilogue warp: NO output sets of NOUT tiles (ping-pong when stores would
  // otherwise stall the next chunk), NA operand sets of NAUX tiles (loads NA chunks ahead),
  // and for the split SwiGLU the round(a) tiles of the warp's chunks.
  // Split-phase kinds stage h and b (a is staged in the round(a) tiles); the h-only SwiGLU stages h.
  static constexpr int OSET = (SPLIT ? (K == EPI_SWIGLU_H ? 1 : 2) : D::NOUT) * OUT_BUF;
  static constexpr int ASET = D::NAUX * AUX_BUF;
  static constexpr int ABUF = SPLIT ? (BN / CW / 2) * OUT_BUF : 0;
  // The three-accumulator kernel uses one set of da, db tiles: its shared memory goes to a fourth
  // operand stage, which is worth more (the MMA waits less for operands) than overlapping a chunk's
  // staging with the previous chunk's stores.
  // So does the dsilu epilogue that also writes z (two output tiles per set): one set keeps its five stages.
  static constexpr int NO = (TRIPLE || K == EPI_DSILU_Z) ? 1 : (D::NAUX > 0 || SPLIT) ? 2 : 1;
  static constexpr int NA = D::NAUX > 0 ? aux_sets(K) : 0;
  static constexpr int WARP_BYTES = NO * OSET + NA * ASET + ABUF;
  static constexpr int EPI_BYTES = kEpiWarps * WARP_BYTES;
  // Online RMSNorm: four extra warps accumulate the row sums of squares of the x tiles in the ring.
  static constexpr bool STATS = (K == EPI_NORM_SILU || K == EPI_F32_SS);
  // First epilogue warp: 4 with the register split (warpgroup-aligned epilogue), 2 without.
  static constexpr bool REGSPLIT = !STATS;
  static constexpr int EPI0 = REGSPLIT ? 4 : 2;
  static constexpr int THREADS = 32 * (EPI0 + kEpiWarps) + (STATS ? 128 : 0);
  static constexpr int BAR_BYTES = 1024 + 1024;  // barriers, then s for two tiles of 128 rows
  static constexpr int RING_BUDGET = kMaxSmem - 1024 - EPI_BYTES - BAR_BYTES;
  static constexpr int STAGES = RING_BUDGET / STAGE_BYTES > 8 ? 8 : RING_BUDGET / STAGE_BYTES;
  static constexpr uint32_t TMEM_COLS = NBUF * ACC_COLS <= 32    ? 32
                                        : NBUF * ACC_COLS <= 64  ? 64
                                        : NBUF * ACC_COLS <= 128 ? 128
                                        : NBUF * ACC_COLS <= 256 ? 256
                                                                 : 512;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_BYTES + BAR_BYTES;
  static_assert(NBUF * ACC_COLS <= 512, "accumulator buffers must fit in TMEM");
  static_assert(STAGES >= 2, "need at least two stages");
  static_assert(BN % 128 == 0 && BN <= 256, "BN must be 128 or 256 (each CTA stages BN/2, whole 64-column chunks)");
  static_assert((BN / CW) % 2 == 0, "both epilogue warps of a lane quarter need the same number of chunks");
  static_assert(OSET % 1024 == 0 || (OSET % 512 == 0 && !D::OUT_F32), "staging tiles keep swizzle alignment");
  static_assert(ASET % 512 == 0 && ABUF % 512 == 0, "staging tiles keep swizzle alignment");
  static_assert(NA <= kMaxAuxSets, "operand-tile barriers per warp");
  static_assert(NACC <= kMaxAcc, "accumulator barriers");
  static_assert(3 * 8 + kMaxAcc + kMaxAcc + 1 + kMaxAuxSets * kEpiWarps + 2 + 2 <= 127,
                "barriers, TMEM slot and flag fit");
  static_assert(SMEM_BYTES <= kMaxSmem, "shared memory budget");
};

// Pair-tile index -> (split, batch, this CTA's m-tile, n-tile); n runs fastest.
// K blocks of the tile in CTA row block mb (split range, narrowed by a causal mask: mode 2 drops keys
// past the pair tile's last query, mode 3 queries before its first key).
__device__ __forceinline__ void k_range(const Shape& sh, int split, int mb, int& kb0, int& kb1) {
  kb0 = split * sh.kb_per_split;
  kb1 = min(sh.kb_total, kb0 + sh.kb_per_split);
  const int row0 = (mb >> 1) * 2 * BM;  // first row of the pair tile
  if (sh.causal == 2) kb1 = min(kb1, (row0 + 2 * BM) / BK);
  if (sh.causal == 3) kb0 = max(kb0, row0 / BK);
}

// Where batch `batch` of a row-batched problem starts in each tensor (all 0 otherwise).  RB: the
// kernel is built for row-batched problems (the per-batch offsets and the causal tile schedule
// exist only there, so the other kernels carry none of that code).
struct BatchOff {
  int ra, ca, rb, cb, ro, co;  // stored row and column of A, B and the output
};
template <bool RB>
__device__ __forceinline__ BatchOff batch_off(const Shape& sh, int batch) {
  if (!RB || !sh.rowbatch) return BatchOff{0, 0, 0, 0, 0, 0};
  const int hi = batch / sh.bh, lo = batch - hi * sh.bh;
  return BatchOff{hi * sh.rb_a + lo * sh.rl_a, lo * sh.cb_a, hi * sh.rb_b + lo * sh.rl_b,
                  lo * sh.cb_b, hi * sh.rb_o + lo * sh.rl_o, lo * sh.cb_o};
}

// Pair tiles of one batch.  Causal mode 1 (M = N) schedules only the tiles on or below the
// diagonal: pair p (rows 256 p .. 256 p + 255) takes its first (p + 1) u key tiles, u = 256 / BN.
template <bool RB>
__host__ __device__ __forceinline__ int batch_tiles(const Shape& sh) {
  if (RB && sh.causal == 1) return sh.n_tiles / sh.m_pairs * (sh.m_pairs * (sh.m_pairs + 1) / 2);
  return sh.m_pairs * sh.n_tiles;
}

template <bool RB>
__host__ __device__ __forceinline__ void decode_tile(const Shape& sh, int tile, int rank, int& split, int& batch, int& mb,
                                            int& nb) {
  if (sh.grouped) {
    const int per_split = sh.g_tiles;
    if (sh.reverse) tile = sh.ksplit * per_split - 1 - tile;
    split = tile / per_split;
    int rem = tile - split * per_split;
    // The batch whose tile range holds rem (constant indices only: the shape stays in registers).
    int b = 0, t0 = 0, nt = sh.g_n_tiles[0];
#pragma unroll
    for (int i = 1; i < kMaxBatch; ++i) {
      if (i < sh.batches && rem >= sh.g_tile0[i]) {
        b = i;
        t0 = sh.g_tile0[i];
        nt = sh.g_n_tiles[i];
      }
    }
    batch = b;
    rem -= t0;
    const int mp = rem / nt;
    nb = rem - mp * nt;
    mb = 2 * mp + rank;
    return;
  }
  const int per_batch = batch_tiles<RB>(sh);
  const int per_split = sh.batches * per_batch;
  if (sh.reverse) tile = sh.ksplit * per_split - 1 - tile;
  split = tile / per_split;
  int rem = tile - split * per_split;
  batch = rem / per_batch;
  rem -= batch * per_batch;
  if (RB && sh.causal == 1) {
    const int u = sh.n_tiles / sh.m_pairs;  // key tiles per pair of query tiles
    const int q = rem / u;                  // pair p holds q in [p (p + 1) / 2, (p + 1) (p + 2) / 2)
    int p = static_cast<int>((sqrtf(8.f * q + 1.f) - 1.f) * 0.5f);
    while ((p + 1) * (p + 2) / 2 <= q) ++p;
    while (p > 0 && p * (p + 1) / 2 > q) --p;
    nb = rem - u * (p * (p + 1) / 2);
    mb = 2 * p + rank;
    return;
  }
  int mp = rem / sh.n_tiles;
  nb = rem - mp * sh.n_tiles;
  if (RB && (sh.causal == 2 || sh.causal == 3)) {
    // Causal K ranges grow (mode 2) or shrink (mode 3) with the row block.  Within a batch the row
    // blocks are taken as 0, 1, .., m/2 - 1, then m - 1, m - 2, .., m/2, so that tiles m/2 apart in the
    // launch order (as a pair's round-robin share is when the pair count is an odd multiple of m/2) have
    // complementary lengths; a batch's tiles stay together (its K operand in L2).
    const int h = sh.m_pairs >> 1;
    if (mp >= h) mp = sh.m_pairs - 1 - (mp - h);
  }
  mb = 2 * mp + rank;
}

template <EpiKind K, int BN, bool A_MN, bool B_MN, bool RB>
__global__ void __launch_bounds__(Config<K, BN>::THREADS, 1)
    gemm_kernel(const __grid_constant__ Maps maps, const Shape sh, const EpiParams ep) {
  using C = Config<K, BN>;
  using D = EpiDef<K>;
  constexpr int NACC = D::NACC;
  constexpr int STAGES = C::STAGES;
  constexpr uint32_t IDESC = idesc_bf16<BN, A_MN, B_MN>();
  constexpr uint32_t IDESC_BMN = idesc_bf16<BN, A_MN, true>();  // sets in C::B_MN_SETS

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint8_t* sE = sB + STAGES * C::B_BYTES;  // epilogue staging, 1024-aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(sE + C::EPI_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* consumed = empty + STAGES;  // MMA done with a stage (statistics warps may read it)
  uint64_t* tfull = consumed + STAGES;
  uint64_t* tempty = tfull + kMaxAcc;
  uint64_t* drain = tempty + kMaxAcc;
  uint64_t* aux_full = drain + 1;                       // per epilogue warp and operand set
  uint64_t* sfull = aux_full + kMaxAuxSets * kEpiWarps;  // stats -> epilogue, per TMEM buffer
  uint64_t* sempty = sfull + 2;     // epilogue -> stats, per TMEM buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* s_rows = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(full) + 1024);  // [2][BM]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full[i], 1);                  // leader: its producer's expect_tx (+ both CTAs' bytes)
      mbar_init(&empty[i], C::STATS ? 4 : 1);  // MMA commit, or the statistics warps after it
      mbar_init(&consumed[i], 1);
    }
    for (int i = 0; i < kMaxAcc; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 2 * kEpiWarps);  // leader: one arrive per epilogue warp of both CTAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 4);
      mbar_init(&sempty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < kMaxAuxSets * kEpiWarps; ++i) mbar_init(&aux_full[i], 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
  }
  if (warp == 0 && lane == 0) {
    const int nsets = NACC > 1 ? NACC : (sh.rowbatch ? 1 : sh.batches);
    for (int i = 0; i < nsets; ++i) {
      tmap_prefetch(&maps.a[i]);
      tmap_prefetch(&maps.b[i]);
    }
  }
  __syncwarp();
  if (warp == 1) tmem_alloc(tmem_slot, C::TMEM_COLS);  // both CTAs: one joint allocation
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers and TMEM exist before either touches the other
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above touches no global memory; it overlaps the previous kernel's tail.
  pdl_wait();

  const int rank = static_cast<int>(blockIdx.x & 1);  // 0: leader (issues the MMAs)
  const int cid = static_cast<int>(blockIdx.x >> 1);
  const int ncl = static_cast<int>(gridDim.x >> 1);
  constexpr uint16_t kBoth = 0x3;
  const int total =  // pair tiles
      sh.ksplit * (sh.grouped ? sh.g_tiles : sh.batches * batch_tiles<RB>(sh));

  // Each warpgroup's branch starts with its share of the register split (setmaxnreg; the launcher
  // checks that the split fits the launch's registers before launching).
  if (warp < C::EPI0) {
    if constexpr (C::REGSPLIT) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegCtl));
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer
        int st = 0;
        uint32_t ph = 0;
        long long issued = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += ncl) {
          int split, batch, mb, nb;
          decode_tile<RB>(sh, tile, rank, split, batch, mb, nb);
          int kb0, kb1;
          k_range(sh, split, mb, kb0, kb1);
          const int m0 = mb * BM, n0 = nb * BN;
          const int set0 = sh.rowbatch ? 0 : batch;
          const BatchOff bo = batch_off<RB>(sh, batch);
          for (int s = 0; s < NACC && ok; ++s) {
            const int set = NACC > 1 ? s : set0;
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait(&empty[st], ph ^ 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_PRODUCER)) {
                ok = false;
                break;
              }
              // The leader's full barrier counts the bytes of both CTAs' halves of the stage.
              if (rank == 0) mbar_expect_tx(&full[st], 2 * C::STAGE_BYTES);
              const uint32_t fbar = mapa(smem_addr(&full[st]), 0);
              uint8_t* a_dst = sA + st * C::A_BYTES;
              uint8_t* b_dst = sB + st * C::B_BYTES;
              if (A_MN) {
  #pragma unroll
                for (int j = 0; j < BM / 64; ++j)
                  tma_load_2d_pair(a_dst + j * 8192, &maps.a[set], fbar, m0 + 64 * j + bo.ca, kb * BK + bo.ra);
              } else {
                tma_load_2d_pair(a_dst, &maps.a[set], fbar, kb * BK + bo.ca, m0 + bo.ra);
              }
              const int nb0 = n0 + rank * (BN / 2);  // this CTA's half of the B tile
              if (B_MN || ((C::B_MN_SETS >> set) & 1u)) {
  #pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                  tma_load_2d_pair(b_dst + j * 8192, &maps.b[set], fbar, nb0 + 64 * j + bo.cb, kb * BK + bo.rb);
              } else {
                tma_load_2d_pair(b_dst, &maps.b[set], fbar, kb * BK + bo.cb, nb0 + bo.rb);
              }
              ++issued;
              if (++st == STAGES) {
                st = 0;
                ph ^= 1u;
              }
            }
          }
        }
        pdl_trigger();  // every load of this CTA is issued: the next kernel may be scheduled
        if (!ok && rank == 0) {
          // Wait (bounded) for the pair's copies still in flight before the CTAs may exit.
          const long long n_back = issued < STAGES ? issued : STAGES;
          for (long long i = 1; i <= n_back; ++i) {
            const long long n = issued - i;
            const int s = static_cast<int>(n % STAGES);
            const uint32_t p = static_cast<uint32_t>((n / STAGES) & 1);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_test(&full[s], p) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer (leader CTA)
        const uint32_t a_base = smem_addr(sA);
        const uint32_t b_base = smem_addr(sB);
        int st = 0;
        uint32_t ph = 0;
        int it = 0;
        bool ok = true;
        uint32_t ruse[2] = {0u, 0u};  // TRIPLE: accumulations started in each TMEM region
        for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
          int split, batch, mb, nb;
          decode_tile<RB>(sh, tile, rank, split, batch, mb, nb);
          int kb0, kb1;
          k_range(sh, split, mb, kb0, kb1);
          const int buf = C::NBUF == 2 ? (it & 1) : 0;
          const uint32_t tph = static_cast<uint32_t>(C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1));
          if (!C::SPLIT) {
            if (!mbar_wait(&tempty[buf], tph ^ 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          for (int s = 0; s < NACC && ok; ++s) {
            // Split-phase kernels: accumulator s lives in region reg (its own full / empty pair).
            const int reg = C::TRIPLE ? (s == 1 ? 1 - (it & 1) : (it & 1)) : s;
            if (C::SPLIT) {
              const uint32_t uph = C::TRIPLE ? (ruse[reg] & 1u) : tph;
              if (!mbar_wait(&tempty[reg], uph ^ 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_MMA)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + buf * C::ACC_COLS + reg * BN;
            for (int kb = kb0; kb < kb1; ++kb) {
              if (!mbar_wait(&full[st], ph, abort_flag, sh.err, DEV_ERR_TIMEOUT_MMA)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t a_st = a_base + st * C::A_BYTES;
              const uint32_t b_st = b_base + st * C::B_BYTES;
  #pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                // K-major: the 16-wide K slice sits 32 bytes further along each swizzled 128-byte row.
                // MN-major: it is 16 rows (2 atoms of 8 rows x 128 bytes) further on.
                const uint64_t ad = A_MN ? sdesc(a_st + kk * 2048, 8192, 1024) : sdesc(a_st + kk * 32, 16, 1024);
                const bool bmn = B_MN || ((C::B_MN_SETS >> s) & 1u);
                const uint64_t bd = bmn ? sdesc(b_st + kk * 2048, 8192, 1024) : sdesc(b_st + kk * 32, 16, 1024);
                umma_f16(d_tmem, ad, bd, bmn ? IDESC_BMN : IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
              }
              // Both CTAs' halves of the stage are free once these MMAs complete.
              umma_commit(C::STATS ? &consumed[st] : &empty[st], kBoth);
              if (++st == STAGES) {
                st = 0;
                ph ^= 1u;
              }
            }
            if (C::SPLIT && ok) {
              umma_commit(&tfull[reg], kBoth);
              if (C::TRIPLE) ++ruse[reg];
            }
          }
          if (!C::SPLIT && ok) umma_commit(&tfull[buf], kBoth);
        }
        // Drain: all MMAs issued by this thread have completed once this barrier flips.
        umma_commit(drain, 0x1);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(drain, 0) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }  // with the register split, warps 2 and 3 are idle
  } else if (C::STATS && warp >= C::EPI0 + kEpiWarps) {
    // ------------------------------------------------ online-RMSNorm statistics warps
    // Row r of the x tile is 128 bytes per stage with its 16-byte chunks permuted by the
    // swizzle; a sum of squares over the whole row does not depend on that order, and
    // reading logical chunk j at physical position j ^ (r & 7) keeps the 8-thread phases
    // of each 16-byte shared load on distinct banks.
    const int row = (warp - C::EPI0 - kEpiWarps) * 32 + lane;
    int st = 0;
    uint32_t ph = 0;
    int it = 0;
    bool ok = true;
    for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
      int split, batch, mb, nb;
      decode_tile<RB>(sh, tile, rank, split, batch, mb, nb);
      int kb0, kb1;
      k_range(sh, split, mb, kb0, kb1);
      float ss = 0.f;
      for (int kb = kb0; kb < kb1; ++kb) {
        // The MMAs have read the stage of both CTAs (so it has landed); it is refilled only
        // after these warps arrive on `empty`.
        if (!mbar_wait(&consumed[st], ph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE)) {
          ok = false;
          break;
        }
        const uint8_t* a_row = sA + st * C::A_BYTES + row * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float v[8];
          lds_bf16x8(smem_addr(a_row) + ((j ^ (row & 7)) << 4), v);
#pragma unroll
          for (int t = 0; t < 8; ++t) ss = fmaf(v[t], v[t], ss);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
        if (++st == STAGES) {
          st = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      const float s_val = rsqrtf(ss * ep.coef + ep.eps);
      const int m = mb * BM + row;
      // The 1/rms row scale, or for a row-parallel partial the raw sum of squares of its shard.
      if (nb == 0 && m < sh.M && ep.rowscale_out) ep.rowscale_out[m] = K == EPI_F32_SS ? ss : s_val;
      const int buf = it & 1;
      const uint32_t tph = static_cast<uint32_t>((it >> 1) & 1);
      if (!mbar_wait(&sempty[buf], tph ^ 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE)) break;
      s_rows[buf * BM + row] = s_val;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfull[buf]);
    }
  } else {
    if constexpr (C::REGSPLIT) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegEpi));
    // ------------------------------------------------ epilogue warps
    // Each epilogue warp is an independent unit: warp (g, q) owns TMEM lane quarter q (rows
    // 32 q .. 32 q + 31 of the CTA's tile) and the chunks c = g, g+2, ... of each tile.  Its
    // lane 0 loads the chunk's operand tiles and stores its output tiles (32 x 32 boxes)
    // through the warp's own staging sets; the warp synchronises only with itself.
    constexpr int NAUX = D::NAUX, NOUT = D::NOUT;
    constexpr int NCH = BN / CW;
    constexpr int NO = C::NO, NA = C::NA;
    const int ew = warp - C::EPI0;
    const int g = ew >> 2;   // chunk parity
    const int q = warp & 3;  // TMEM lane quarter this warp may access (warp id mod 4)
    const int row = q * 32 + lane;
    const bool leader = lane == 0;
    uint8_t* wstage = sE + ew * C::WARP_BYTES;  // NO output sets | NA operand sets | round(a) tiles
    auto ostage = [&](int b) { return wstage + b * C::OSET; };
    auto astage = [&](int b) { return wstage + NO * C::OSET + b * C::ASET; };
    uint64_t* abar = &aux_full[kMaxAuxSets * ew];
    uint32_t aph = 0u;      // bit b: phase parity of abar[b]
    uint32_t pending = 0u;  // lane 0, bit b: an operand-tile load is in flight on abar[b]

    // The warp's chunk sequence: (tile, c) for c = g, g+2, ... of each of this CTA's tiles.
    auto next_chunk = [&](int& t, int& c) {
      c += 2;
      if (c >= NCH) {
        t += ncl;
        c = g;
      }
    };
    auto issue_aux = [&](int t, int c, int b) {
      int split, batch, mb, nb;
      decode_tile<RB>(sh, t, rank, split, batch, mb, nb);
      uint32_t bytes = 0;
#pragma unroll
      for (int a = 0; a < NAUX; ++a)
        if (epi_aux_ptr(ep, a, batch)) bytes += C::AUX_BUF;
      mbar_expect_tx(&abar[b], bytes);
#pragma unroll
      for (int a = 0; a < NAUX; ++a)
        if (epi_aux_ptr(ep, a, batch))
          tma_load_2d(astage(b) + a * C::AUX_BUF, &maps.aux[batch][a], &abar[b], nb * BN + c * CW,
                      mb * BM + q * ER);
      pending |= 1u << b;
    };
    // Lane 0: the stores that last used output set b have finished reading it.
    auto wait_set_free = [&]() {
      if (leader) {
        asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(NO - 1) : "memory");
      }
    };
    // Prefetch cursor: the next chunk whose operand tiles are not yet requested.
    int pf_t = cid, pf_c = g;
    if constexpr (NAUX > 0) {
      if (leader) {
        for (int b = 0; b < NA && pf_t < total; ++b) {
          issue_aux(pf_t, pf_c, b);
          next_chunk(pf_t, pf_c);
        }
      }
    }

    bool ok = true;
    int it = 0;
    int qi = 0;  // index of the warp's current chunk in its sequence
    uint32_t euse[2] = {0u, 0u};  // TRIPLE: accumulations consumed from each TMEM region
    for (int tile = cid; tile < total && ok; tile += ncl, ++it) {
      int split, batch, mb, nb;
      decode_tile<RB>(sh, tile, rank, split, batch, mb, nb);
      const int buf = C::NBUF == 2 ? (it & 1) : 0;
      const uint32_t tph = static_cast<uint32_t>(C::NBUF == 2 ? ((it >> 1) & 1) : (it & 1));
      const int sbuf = it & 1;  // statistics double buffer (independent of TMEM)
      const uint32_t sph = static_cast<uint32_t>((it >> 1) & 1);
      const int m = mb * BM + row;
      const int ob = sh.rowbatch ? 0 : batch;                 // output maps and pointers of this batch
      const BatchOff bo = batch_off<RB>(sh, batch);
      const int r0 = mb * BM + q * ER + bo.ro;  // first stored row of this warp's boxes
      const int x0 = nb * BN + bo.co;           // first stored column of the tile
      // Causal mode 1: a tile wholly above the diagonal (every column past every row) is not stored
      // (the schedule holds none; the test guards the stores all the same).
      const bool no_store = sh.causal == 1 && nb * BN >= (mb >> 1) * 2 * BM + 2 * BM;
      RowIn ri;
      if constexpr (C::STATS) {
        ri.k = 0.f;
        ri.act = ep.act;
        ok = mbar_wait(&sfull[sbuf], sph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE);
        ri.s = s_rows[sbuf * BM + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[sbuf]);
      } else {
        ri = row_inputs<K>(ep, m);
      }
      bool present[NOUT];
#pragma unroll
      for (int o = 0; o < NOUT; ++o) present[o] = epi_out_ptr(ep, o, ob) != nullptr;
      bool aux_present[NAUX > 0 ? NAUX : 1];
#pragma unroll
      for (int a = 0; a < NAUX; ++a) aux_present[a] = epi_aux_ptr(ep, a, ob) != nullptr;

      if constexpr (K == EPI_ATTN_BWD) {
        // Causal attention backward scores.  Phase 1: P = exp(scale S - lse) from accumulator 0
        // (0 where the key is past the query) into the warp's shared-memory tiles and out to P;
        // S's columns are released.  Phase 2: dS = scale P (dP - D) from accumulator 1 (fp32) and
        // those tiles, out to dS; then dP's columns are released.  Tiles wholly above the diagonal
        // only pass their accumulators back.
        constexpr int NC = NCH / 2;
        constexpr float kLog2e = 1.4426950408889634f;
        uint8_t* abuf = wstage + NO * C::OSET + NA * C::ASET;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        const int grow = m + bo.ro;  // lse and D are indexed like the output's rows
        const bool row_in = m < sh.M;
        const float lse2 = row_in ? ep.rowscale[grow] * kLog2e : 0.f;
        const float dval = row_in ? ep.rowpart_in[grow] : 0.f;
        const float c2 = ep.coef * kLog2e;
        ok = mbar_wait(&tfull[0], tph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        tc_fence_after();
        if (!no_store) {
          if (leader) bulk_wait_read_all();  // the previous tile's P stores have read abuf
          __syncwarp();
#pragma unroll
          for (int ci = 0; ci < NC; ++ci) {
            const int c = g + 2 * ci;
            float v[CW];
            tmem_ld32(t_row + c * CW, v);
            tmem_ld_wait();
            const int n0 = nb * BN + c * CW;
#pragma unroll
            for (int j = 0; j < CW; ++j) v[j] = (n0 + j <= m && row_in) ? exp2f(v[j] * c2 - lse2) : 0.f;
            const uint32_t base = smem_addr(abuf + ci * C::OUT_BUF);
#pragma unroll
            for (int j = 0; j < CW / 8; ++j) sts_bf16x8(base + stage_off<64>(lane, j), &v[8 * j]);
          }
          fence_async_smem();
          __syncwarp();
          if (leader && present[0]) {
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
              tma_store_2d(&maps.out[ob][0], abuf + ci * C::OUT_BUF, x0 + (g + 2 * ci) * CW, r0);
            bulk_commit();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[0]), 0));
        ok = mbar_wait(&tfull[1], tph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        tc_fence_after();
        if (!no_store) {
#pragma unroll 1
          for (int ci = 0; ci < NC; ++ci) {
            const int c = g + 2 * ci;
            const int b = qi % NO;
            wait_set_free();
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            float v[CW];
            tmem_ld32(t_row + BN + c * CW, v);
            tmem_ld_wait();
            const uint32_t abase = smem_addr(abuf + ci * C::OUT_BUF);
            const uint32_t dbase = smem_addr(ostage(b));
#pragma unroll
            for (int j = 0; j < CW / 8; ++j) {
              float p[8], d8[8];
              lds_bf16x8(abase + stage_off<64>(lane, j), p);
#pragma unroll
              for (int t = 0; t < 8; ++t) d8[t] = ep.coef * p[t] * (v[8 * j + t] - dval);
              sts_bf16x8(dbase + stage_off<64>(lane, j), d8);
            }
            fence_async_smem();
            __syncwarp();
            if (leader) {
              if (present[1]) tma_store_2d(&maps.out[ob][1], ostage(b), x0 + c * CW, r0);
              bulk_commit();
            }
            ++qi;
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[1]), 0));
        if (!ok) break;
      } else if constexpr (C::TRIPLE) {
        // Checkpointed re-forward and SwiGLU backward of one tile.  The accumulators are a (z_g
        // B_gate^T), b (z_u B_up^T) and dh (du_down A_down), in that MMA order; a and dh take region
        // it mod 2 of TMEM, b the other.  Phase 1 stages round(a) in shared memory and releases its
        // region (dh accumulates there next); phase 2 packs round(b) into registers and releases
        // its region (the next tile's a); phase 3 reads dh chunk by chunk, releasing the region
        // after the last load, and forms h = SiLU(a) b, da = dh b SiLU'(a), db = dh SiLU(a) (the
        // expressions of the forward SwiGLU and of the separate SwiGLU backward: both paths give
        // the same bits).  h is written over the chunk's a tile and stored from there; da, db go
        // through the two output sets.
        constexpr int NC = NCH / 2;
        uint8_t* abuf = wstage + NO * C::OSET + NA * C::ASET;
        const int r0g = it & 1, r1g = 1 - r0g;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        ok = mbar_wait(&tfull[r0g], euse[r0g] & 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        ++euse[r0g];
        tc_fence_after();
        if (leader) bulk_wait_read_all();  // the previous tile's h stores have read the a tiles
        __syncwarp();
        static_assert(NC % 2 == 0, "phases 1 and 2 load two chunks per TMEM wait");
#pragma unroll
        for (int ci = 0; ci < NC; ci += 2) {  // two chunks per wait: the load latency is paid half as often
          float v[2][CW];
          tmem_ld32(t_row + r0g * BN + (g + 2 * ci) * CW, v[0]);
          tmem_ld32(t_row + r0g * BN + (g + 2 * ci + 2) * CW, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t base = smem_addr(abuf + (ci + u) * C::OUT_BUF);
#pragma unroll
            for (int j = 0; j < CW / 8; ++j) sts_bf16x8(base + stage_off<64>(lane, j), &v[u][8 * j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[r0g]), 0));
        uint32_t bpk[NC][CW / 2];
        ok = mbar_wait(&tfull[r1g], euse[r1g] & 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        ++euse[r1g];
        tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < NC; ci += 2) {
          float v[2][CW];
          tmem_ld32(t_row + r1g * BN + (g + 2 * ci) * CW, v[0]);
          tmem_ld32(t_row + r1g * BN + (g + 2 * ci + 2) * CW, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
#pragma unroll
            for (int j = 0; j < CW / 2; ++j) bpk[ci + u][j] = pack_bf16x2(v[u][2 * j], v[u][2 * j + 1]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[r1g]), 0));
        ok = mbar_wait(&tfull[r0g], euse[r0g] & 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        ++euse[r0g];
        tc_fence_after();
        // dh is read 16 columns at a time (register pressure), each piece's load issued before the
        // arithmetic on the previous one.
        float dhb[2][CW / 2];
        tmem_ld16(t_row + r0g * BN + g * CW, dhb[0]);
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          const int c = g + 2 * ci;
          const uint32_t abase = smem_addr(abuf + ci * C::OUT_BUF);
          // The chunk's h goes over its own a tile at once; da and db wait in registers (packed bf16)
          // until the output set is free, so that wait overlaps this chunk's arithmetic.
          uint32_t dap[CW / 8][4], dbp[CW / 8][4];
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            tmem_ld_wait();
            if (ci == NC - 1 && hh == 1) {  // every dh column of this warp is in registers: region free
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[r0g]), 0));
            } else {
              const int nc = hh == 1 ? c + 2 : c;  // the next piece: this chunk's second half or the next chunk's first
              tmem_ld16(t_row + r0g * BN + nc * CW + (1 - hh) * (CW / 2), dhb[hh ^ 1]);
            }
            const float* dh = dhb[hh];
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
              const int j = 2 * hh + jj;
              float av[8], hv[8], dav[8], dbv[8];
              lds_bf16x8(abase + stage_off<64>(lane, j), av);
#pragma unroll
              for (int t = 0; t < 8; ++t) {
                float b0, b1;
                unpack_bf16x2(bpk[ci][4 * j + t / 2], b0, b1);
                const float bv = (t & 1) ? b1 : b0;
                const float a = av[t], d = dh[8 * jj + t];
                const float l = Num<bf16>::logistic(a);
                hv[t] = silu<bf16>(a) * bv;
                dav[t] = d * bv * (l * (1.f + a * (1.f - l)));
                dbv[t] = d * (a * l);
              }
              sts_bf16x8(abase + stage_off<64>(lane, j), hv);  // over this lane's own a values
#pragma unroll
              for (int t = 0; t < 4; ++t) {
                dap[j][t] = pack_bf16x2(dav[2 * t], dav[2 * t + 1]);
                dbp[j][t] = pack_bf16x2(dbv[2 * t], dbv[2 * t + 1]);
              }
            }
          }
          wait_set_free();
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) {
            tmem_ld_wait();  // the next piece's load may be in flight
            break;
          }
          const int b = qi % NO;
          const uint32_t dbase = smem_addr(ostage(b));
#pragma unroll
          for (int j = 0; j < CW / 8; ++j) {
            sts128(dbase + stage_off<64>(lane, j), dap[j][0], dap[j][1], dap[j][2], dap[j][3]);
            sts128(dbase + C::OUT_BUF + stage_off<64>(lane, j), dbp[j][0], dbp[j][1], dbp[j][2], dbp[j][3]);
          }
          fence_async_smem();
          __syncwarp();
          if (leader) {
            if (present[0]) tma_store_2d(&maps.out[ob][0], abuf + ci * C::OUT_BUF, x0 + c * CW, r0);
            if (present[1]) tma_store_2d(&maps.out[ob][1], ostage(b), x0 + c * CW, r0);
            if (present[2]) tma_store_2d(&maps.out[ob][2], ostage(b) + C::OUT_BUF, x0 + c * CW, r0);
            bulk_commit();
          }
          ++qi;
        }
        if (!ok) break;
      } else if constexpr (C::SPLIT) {
        // Phase 1: round(a) of this warp's chunks into its a tiles in shared memory (exact:
        // a is stored rounded), optionally TMA-stored from there; then a's TMEM columns are
        // released, so the next tile's a accumulation overlaps the rest of this epilogue.
        constexpr int NC = NCH / 2;
        uint8_t* abuf = wstage + NO * C::OSET + NA * C::ASET;  // NC tiles of 32 rows x 32 columns
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
        ok = mbar_wait(&tfull[0], tph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        tc_fence_after();
        constexpr bool OUT_AB = D::NOUT == 3;  // a and b are outputs of the kind (when present)
        if (OUT_AB && present[OUT_AB ? 1 : 0] && leader) bulk_wait_read_all();  // the previous a stores have read abuf
        __syncwarp();
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          const int c = g + 2 * ci;
          float v[CW];
          tmem_ld32(t_row + c * CW, v);
          tmem_ld_wait();
          if constexpr (D::NEED_S) {  // dense gate/up: the 1/rms row scale of the normalised input
#pragma unroll
            for (int j = 0; j < CW; ++j) v[j] *= ri.s;
          }
          const uint32_t base = smem_addr(abuf + ci * C::OUT_BUF);
#pragma unroll
          for (int j = 0; j < CW / 8; ++j) sts_bf16x8(base + stage_off<64>(lane, j), &v[8 * j]);
        }
        if (OUT_AB && present[OUT_AB ? 1 : 0]) {
          fence_async_smem();
          __syncwarp();
          if (leader) {
#pragma unroll
            for (int ci = 0; ci < NC; ++ci)
              tma_store_2d(&maps.out[ob][OUT_AB ? 1 : 0], abuf + ci * C::OUT_BUF, x0 + (g + 2 * ci) * CW, r0);
            bulk_commit();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[0]), 0));
        // Phase 2a: round(b) of this warp's chunks into registers (packed bf16, exact); then b's
        // columns are released and the next tile's b accumulation overlaps the h math and stores.
        uint32_t bpk[NC][CW / 2];
        ok = mbar_wait(&tfull[1], tph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        tc_fence_after();
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          float v[CW];
          tmem_ld32(t_row + BN + (g + 2 * ci) * CW, v);
          tmem_ld_wait();
          if constexpr (D::NEED_S) {
#pragma unroll
            for (int j = 0; j < CW; ++j) v[j] *= ri.s;
          }
#pragma unroll
          for (int j = 0; j < CW / 2; ++j) bpk[ci][j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[1]), 0));
        // Phase 2b: h = SiLU(a) b; outputs h and (optionally) b.
#pragma unroll
        for (int ci = 0; ci < NC; ++ci) {
          const int c = g + 2 * ci;
          const int b = qi % NO;
          wait_set_free();
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const uint32_t abase = smem_addr(abuf + ci * C::OUT_BUF);
          const uint32_t hbase = smem_addr(ostage(b));
          const uint32_t bbase = smem_addr(ostage(b) + C::OUT_BUF);
#pragma unroll
          for (int j = 0; j < CW / 8; ++j) {
            float av[8], hv[8];
            lds_bf16x8(abase + stage_off<64>(lane, j), av);
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              float b0, b1;
              unpack_bf16x2(bpk[ci][4 * j + t], b0, b1);
              hv[2 * t] = silu<bf16>(av[2 * t]) * b0;
              hv[2 * t + 1] = silu<bf16>(av[2 * t + 1]) * b1;
            }
            sts_bf16x8(hbase + stage_off<64>(lane, j), hv);
            if (OUT_AB && present[OUT_AB ? 2 : 0])
              sts128(bbase + stage_off<64>(lane, j), bpk[ci][4 * j], bpk[ci][4 * j + 1], bpk[ci][4 * j + 2],
                     bpk[ci][4 * j + 3]);
          }
          fence_async_smem();
          __syncwarp();
          if (leader) {
            if (present[0]) tma_store_2d(&maps.out[ob][0], ostage(b), x0 + c * CW, r0);
            if (OUT_AB && present[OUT_AB ? 2 : 0])
              tma_store_2d(&maps.out[ob][OUT_AB ? 2 : 0], ostage(b) + C::OUT_BUF, x0 + c * CW, r0);
            bulk_commit();
          }
          ++qi;
        }
        if (!ok) break;
      } else {
        ok = mbar_wait(&tfull[buf], tph, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        tc_fence_after();
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC_COLS;
        // A tile that is not stored (causal mode 1: wholly above the diagonal) skips the chunk work;
        // such launches have no operand tiles, so only this warp's output-set rotation shifts.
#pragma unroll 1
        for (int c = no_store ? NCH : g; c < NCH; c += 2, ++qi) {
          const int b = qi % NO;  // output set
          const int ba = NA > 0 ? qi % NA : 0;  // operand set
          if constexpr (NAUX > 0) {
            const bool landed = mbar_wait(&abar[ba], (aph >> ba) & 1u, abort_flag, sh.err, DEV_ERR_TIMEOUT_EPILOGUE);
            ok = landed && ok;
            if (landed) {
              aph ^= 1u << ba;
              pending &= ~(1u << ba);
            }
          }
          float v[NACC][CW];
#pragma unroll
          for (int a = 0; a < NACC; ++a) tmem_ld32(t_row + a * BN + c * CW, v[a]);
          tmem_ld_wait();
          float av[NAUX > 0 ? NAUX : 1][CW];
#pragma unroll
          for (int a = 0; a < NAUX; ++a) {
            if (aux_present[a]) {
              const uint8_t* base = astage(ba) + a * C::AUX_BUF;
#pragma unroll
              for (int j = 0; j < CW / 8; ++j) lds_bf16x8(smem_addr(base) + stage_off<64>(lane, j), &av[a][8 * j]);
            } else {
#pragma unroll
              for (int j = 0; j < CW; ++j) av[a][j] = 0.f;
            }
          }
          wait_set_free();
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          if constexpr (NAUX > 0) {
            if (leader && pf_t < total) {  // refill the operand set this chunk has just released
              issue_aux(pf_t, pf_c, ba);
              next_chunk(pf_t, pf_c);
            }
          }
          float o[NOUT][CW];
          float part = 0.f;
          D::template run<bf16, CW>(ri, v, av, o, part);
#pragma unroll
          for (int oi = 0; oi < NOUT; ++oi) {
            if (!present[oi]) continue;
            uint8_t* base = ostage(b) + oi * C::OUT_BUF;
            if constexpr (D::OUT_F32) {
#pragma unroll
              for (int j = 0; j < CW / 4; ++j) {
                sts128(smem_addr(base) + stage_off<128>(lane, j), __float_as_uint(o[oi][4 * j]),
                       __float_as_uint(o[oi][4 * j + 1]), __float_as_uint(o[oi][4 * j + 2]),
                       __float_as_uint(o[oi][4 * j + 3]));
              }
            } else {
#pragma unroll
              for (int j = 0; j < CW / 8; ++j) sts_bf16x8(smem_addr(base) + stage_off<64>(lane, j), &o[oi][8 * j]);
            }
          }
          if constexpr (D::ROWPART) {
            const int n0c = nb * BN + c * CW;
            if (m < sh.M && n0c < sh.N)
              ep.rowpart[(static_cast<long long>(batch) * ep.rowpart_chunks + n0c / CW) * sh.M + m] = part;
          }
          fence_async_smem();
          __syncwarp();
          if (leader && !no_store) {
#pragma unroll
            for (int oi = 0; oi < NOUT; ++oi) {
              if (!present[oi]) continue;
              if constexpr (D::OUT_F32) {
                // Split-K partials are summed by the next kernel: keep them in L2 for it.
                if (sh.ksplit > 1)
                  tma_store_3d_hint(&maps.out[ob][oi], ostage(b) + oi * C::OUT_BUF, x0 + c * CW, r0, split,
                                    l2_evict_last());
                else
                  tma_store_3d(&maps.out[ob][oi], ostage(b) + oi * C::OUT_BUF, x0 + c * CW, r0, split);
              }
              else
                tma_store_2d(&maps.out[ob][oi], ostage(b) + oi * C::OUT_BUF, x0 + c * CW, r0);
            }
            bulk_commit();
          }
        }
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa(smem_addr(&tempty[buf]), 0));  // the leader's MMA reuses it
      }
    }
    if (leader) {
      bulk_wait_all();
      for (int b = 0; b < NA; ++b) {  // abort path: let operand-tile loads in flight land before the CTA exits
        if (!((pending >> b) & 1u)) continue;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(&abar[b], (aph >> b) & 1u) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  }

  __syncwarp();
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other may still use its memory or barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_free(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace umma
}  // namespace lr
