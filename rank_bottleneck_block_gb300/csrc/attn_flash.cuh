// Pieces shared by the tcgen05 attention kernels without materialised scores (forward and backward):
// instruction descriptors, single-CTA MMA issue with A from shared memory or TMEM, TMEM stores, the
// element-wise warps' named barrier and the head-grouped order of work items.
#pragma once

#include <cuda.h>

#include "umma_launch.cuh"

namespace lr {
namespace flash {

using umma::bulk_commit;
using umma::bulk_wait_all;
using umma::fence_async_smem;
using umma::mbar_arrive;
using umma::mbar_expect_tx;
using umma::mbar_init;
using umma::mbar_test;
using umma::mbar_wait;
using umma::pack_bf16x2;
using umma::sdesc;
using umma::smem_addr;
using umma::sts128;
using umma::tc_fence_after;
using umma::tc_fence_before;
using umma::tma_load_2d;
using umma::tma_store_2d;
using umma::tmem_ld32;
using umma::tmem_ld_wait;

constexpr int kRows = 128;     // rows of an MMA tile (M) = keys per key block
constexpr int kDh = 128;       // head width these kernels are built for
constexpr int kTile = kRows * kDh * 2;  // 32 KB: one 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;        // 64 columns (one 128-byte swizzle atom wide)
constexpr int kThreads = 384;
constexpr int kSoftmax0 = 4;   // first of the eight element-wise warps (two warpgroups)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Instruction descriptor of kind::f16, fp32 accumulator, bf16 operands, M = 128 and N columns; B_MN:
// B is MN-major (A is always K-major here: from shared memory, or from TMEM).
template <bool B_MN, int N = kRows>
__host__ __device__ constexpr uint32_t idesc_m128() {
  static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
  return (1u << 4) | (1u << 7) | (1u << 10) | ((B_MN ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(kRows >> 4) << 24);
}

__device__ __forceinline__ void mma1(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void commit1(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 16 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// Byte offset of 16-byte chunk c (8 consecutive columns) of row r in a K-major 128 x 128 tile stored as
// two 64-column halves with the 128-byte swizzle (the TMA box layout and the UMMA descriptor layout).
__device__ __forceinline__ uint32_t kmaj_off(int r, int c) {
  return (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// 2^x by the hardware approximation (results below 2^-126 flush to zero: P is stored as bf16 and summed
// against values of order 1, where such terms do not count).
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Named barrier of the eight element-wise warps.
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// The same barrier, returning the AND of `ok` over the eight warps: every softmax thread takes the
// same branch after it, so an error stops all of them at the same barrier.
__device__ __forceinline__ bool softmax_sync_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

// O += P V with A = P read from TMEM (bf16 pairs packed in 32-bit columns, K-major by construction).
__device__ __forceinline__ void mma1_ta(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers (each thread its lane's 32 values).
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Work item t (in fetch order) of a walk over nheads heads x nb blocks -> (rank, head n).  Items come in
// groups of `group` heads (whose operands stay in L2 while the group is worked on) and by rank inside a
// group; the kernels map rank 0 to their heaviest block, so the last items fetched are light ones.
__host__ __device__ __forceinline__ void item_of(int t, int nheads, int nb, int group, int& rank, int& n) {
  const int per_group = group * nb;
  const int gi = t / per_group, r = t - gi * per_group;
  const int gh = group < nheads - gi * group ? group : nheads - gi * group;
  rank = r / gh;
  n = gi * group + (r - rank * gh);
}

// Heads per group: those whose `bytes_per_head` of streamed operands fit in about 32 MiB of L2.
inline int heads_per_group(long long nheads, long long bytes_per_head) {
  const long long g = (32LL << 20) / (bytes_per_head > 0 ? bytes_per_head : 1);
  return static_cast<int>(g < 1 ? 1 : (g > nheads ? nheads : g));
}

}  // namespace flash
}  // namespace lr
