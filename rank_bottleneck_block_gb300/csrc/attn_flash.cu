// Causal attention forward without materialised scores (tcgen05, dh = 128).
//
// One CTA takes 128 queries of one head (query block i) and walks the key blocks 0 .. i of 128 keys:
//
//   S_j = Q K_j^T                      MMA, fp32 in TMEM (two buffers: S_{j+1} overlaps the softmax of j)
//   P_j = 2^(c S_j - m)                the softmax warps, one thread per query row (a TMEM lane), c = scale
//                                      log2(e); m is the row's running maximum of c S, raised lazily
//   O  += P_j V_j                      MMA, A = P_j (bf16, shared memory), fp32 accumulator in TMEM
//
// with the running row sum l = sum 2^(c S - m).  m is raised only when a block's maximum exceeds it by
// more than 8 (powers of two): P then stays below 2^8 and O, l keep their scale until a real change, at
// which point the row's O (TMEM) and l are multiplied by 2^(m_old - m_new) before the block's P V is
// issued.  Every formula is exact for any m; only overflow limits the laziness.  At the end O / l goes to
// the token-major output and lse = ln 2 (m + log2 l) to the head-major row log-sum-exp the backward reads.
//
// Warps: 0 TMA producer (Q once, then K_j and V_j into a two-stage ring), 1 TMEM allocator and MMA
// issuer (one lane), 2-3 idle, 4-7 softmax / output (warp w reads TMEM lanes 32 (w mod 4) ..).  Shared
// memory: Q, K[2], V[2], P[2], each 128 x 128 bf16 (32 KB) in the 128-byte-swizzled UMMA layouts: Q, K, P
// K-major in two 64-column halves, V MN-major in two 64-key halves of two 64-column chunks.  TMEM: S[2]
// at columns 0 and 128, O at 256.  Every mbarrier wait is bounded (error word, abort flag; each role
// then drains what it issued and TMEM is freed).
#include <cuda.h>

#include "attn_kernels.cuh"
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

constexpr int kRows = 128;     // queries per CTA = keys per block = MMA M = N
constexpr int kDh = 128;       // head width this kernel is built for
constexpr int kTile = kRows * kDh * 2;  // 32 KB: one 128 x 128 bf16 tile
constexpr int kHalf = kTile / 2;        // 64 columns (one 128-byte swizzle atom wide)
constexpr int kThreads = 256;
constexpr int kSoftmax0 = 4;   // first softmax warp
constexpr int kSmem = 1024 + 7 * kTile + 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLazy = 8.f;   // raise the running maximum only past this margin (log2 domain)

struct Maps {
  CUtensorMap q, k, v, o;  // q, k, o: boxes of 64 columns x 128 rows; v: 64 x 64
};

// Instruction descriptor of kind::f16, fp32 accumulator, bf16 operands, M = 128, N = 128.
template <bool B_MN>
__host__ __device__ constexpr uint32_t idesc_m128() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((B_MN ? 1u : 0u) << 16) | (static_cast<uint32_t>(kRows >> 3) << 17) |
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

// Byte offset of 16-byte chunk c (8 consecutive columns) of row r in a K-major 128 x 128 tile stored as
// two 64-column halves with the 128-byte swizzle (the TMA box layout and the UMMA descriptor layout).
__device__ __forceinline__ uint32_t kmaj_off(int r, int c) {
  return (c >> 3) * kHalf + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Named barrier of the four softmax warps.
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    attn_flash_fwd_kernel(const __grid_constant__ Maps maps, int nheads, int H, int s, float scale, float* lse,
                          unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTile;      // [2]
  uint8_t* sV = sK + 2 * kTile;  // [2]
  uint8_t* sP = sV + 2 * kTile;  // [2]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * kTile);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* s_empty = bars + 7;   // [2]
  uint64_t* p_full = bars + 9;    // [2]
  uint64_t* p_empty = bars + 11;  // [2]
  uint64_t* o_done = bars + 13;
  uint64_t* drain = bars + 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 15);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Heaviest query blocks first (block i has i + 1 key blocks).
  const int nqb = s / kRows;
  const int qb = nqb - 1 - static_cast<int>(blockIdx.x) / nheads;
  const int n = static_cast<int>(blockIdx.x) % nheads;
  const int bi = n / H, h = n - bi * H;
  const int nkb = qb + 1;
  const int row0 = bi * s + qb * kRows;  // first token of the query block
  const int col0 = h * kDh;              // first column of the head

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    fence_async_smem();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_addr(tmem_slot))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      bool ok = true;
      int issued = 0;
      mbar_expect_tx(q_full, kTile);
      tma_load_2d(sQ, &maps.q, q_full, col0, row0);
      tma_load_2d(sQ + kHalf, &maps.q, q_full, col0 + 64, row0);
      for (int j = 0; j < nkb && ok; ++j) {
        const int st = j & 1;
        const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
        if (!mbar_wait(&kv_empty[st], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        mbar_expect_tx(&kv_full[st], 2 * kTile);
        const int key0 = bi * s + j * kRows;
        uint8_t* k_dst = sK + st * kTile;
        uint8_t* v_dst = sV + st * kTile;
        tma_load_2d(k_dst, &maps.k, &kv_full[st], col0, key0);
        tma_load_2d(k_dst + kHalf, &maps.k, &kv_full[st], col0 + 64, key0);
        // V as the MN-major B operand: per 64-key half, two 64-column chunks of 64 keys x 128 bytes
        for (int kh = 0; kh < 2; ++kh)
          for (int ch = 0; ch < 2; ++ch)
            tma_load_2d(v_dst + kh * kHalf + ch * (kHalf / 2), &maps.v, &kv_full[st], col0 + 64 * ch, key0 + 64 * kh);
        ++issued;
      }
      // Wait (bounded) for every copy still in flight before the CTA may exit.
      if (!ok) {
        for (int j = (issued > 2 ? issued - 2 : 0); j < issued; ++j) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(&kv_full[j & 1], static_cast<uint32_t>((j >> 1) & 1)) &&
                 global_timer_ns() - t0 < umma::kWaitLimitNs) {
          }
        }
        const uint64_t t0 = global_timer_ns();
        while (!mbar_test(q_full, 0) && global_timer_ns() - t0 < umma::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS = idesc_m128<false>();  // S = Q K^T: both K-major
      constexpr uint32_t kIdO = idesc_m128<true>();   // O += P V: P K-major, V MN-major
      const uint32_t q_base = smem_addr(sQ), k_base = smem_addr(sK), v_base = smem_addr(sV), p_base = smem_addr(sP);
      bool ok = mbar_wait(q_full, 0, abort_flag, err, DEV_ERR_TIMEOUT_MMA);
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1, sb = j & 1;
        const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
        if (!mbar_wait(&s_empty[sb], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) return false;
        if (!mbar_wait(&kv_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) return false;
        tc_fence_after();
        const uint32_t kt = k_base + st * kTile;
#pragma unroll
        for (int kk = 0; kk < kDh / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma1(tmem + sb * kRows, sdesc(q_base + off, 16, 1024), sdesc(kt + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        commit1(&s_full[sb]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkb && ok; ++j) {
        if (j + 1 < nkb && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        const int st = j & 1, pb = j & 1;
        const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
        if (!mbar_wait(&p_full[pb], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pt = p_base + pb * kTile, vt = v_base + st * kTile;
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {  // K = the block's 128 keys
          const uint64_t ad = sdesc(pt + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc(vt + (kk >> 2) * kHalf + (kk & 3) * 2048, kHalf / 2, 1024);
          mma1(tmem + 2 * kRows, ad, bd, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        commit1(o_done);
        commit1(&p_empty[pb]);
        commit1(&kv_empty[st]);
      }
      // Drain: every MMA issued by this thread has completed once this barrier flips.
      commit1(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_test(drain, 0) && global_timer_ns() - t0 < umma::kWaitLimitNs) {
      }
    }
  } else if (warp >= kSoftmax0) {
    // ------------------------------------------------ softmax and output (one thread per query row)
    const int q = warp & 3;
    const int row = q * 32 + lane;  // query row within the block (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const float c = scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkb && ok; ++j) {
      const int sb = j & 1;
      const uint32_t ph = static_cast<uint32_t>((j >> 1) & 1);
      ok = mbar_wait(&s_full[sb], ph, abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      float x[kRows];
#pragma unroll
      for (int cc = 0; cc < kRows / 32; ++cc) tmem_ld32(t_lane + sb * kRows + cc * 32, &x[cc * 32]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[sb]);  // S buffer free for S_{j+2}
      const bool diag = j == qb;
      float bm = -INFINITY;
#pragma unroll
      for (int kk = 0; kk < kRows; ++kk) {
        x[kk] = (diag && kk > row) ? -INFINITY : x[kk] * c;
        bm = fmaxf(bm, x[kk]);
      }
      // Lazy maximum: raise m (and rescale O, l) only when the block's maximum passes it by kLazy.
      const bool raise = m == -INFINITY ? true : bm > m + kLazy;
      const float m_new = raise ? fmaxf(m, bm) : m;
      const float alpha = (raise && m != -INFINITY) ? exp2f(m - m_new) : 1.f;
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds the blocks before j: wait for P_{j-1} V_{j-1}, then scale this row of O.
        const uint32_t op = static_cast<uint32_t>((j - 1) & 1);
        ok = mbar_wait(o_done, op, abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kDh / 32; ++cc) {
          float o[32];
          tmem_ld32(t_lane + 2 * kRows + cc * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] *= alpha;
          tmem_st32(t_lane + 2 * kRows + cc * 32, o);
        }
        tmem_st_wait();
      }
      l *= alpha;
      m = m_new;
      // P into buffer j mod 2 once P_{j-2} V_{j-2} has read it.
      const int pb = j & 1;
      ok = mbar_wait(&p_empty[pb], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE) && ok;
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const uint32_t pt = smem_addr(sP + pb * kTile);
#pragma unroll
      for (int cc = 0; cc < kRows / 8; ++cc) {
        float p[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          p[t] = exp2f(x[8 * cc + t] - m);
          l += p[t];
        }
        sts128(pt + kmaj_off(row, cc), pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]), pack_bf16x2(p[4], p[5]),
               pack_bf16x2(p[6], p[7]));
      }
      fence_async_smem();  // the generic-proxy writes of P become visible to the MMA (async proxy)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[pb]);
    }
    if (ok) {
      // O = O / l after the last P V; stage it in the Q tile (every S MMA has completed) and store.
      ok = mbar_wait(o_done, static_cast<uint32_t>((nkb - 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
      ok = __all_sync(0xffffffffu, ok);
    }
    softmax_sync();  // every softmax warp has decided (each either staged or not)
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l;
      const uint32_t ob = smem_addr(sQ);
#pragma unroll
      for (int cc = 0; cc < kDh / 32; ++cc) {
        float o[32];
        tmem_ld32(t_lane + 2 * kRows + cc * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int g = 0; g < 4; ++g)
          sts128(ob + kmaj_off(row, cc * 4 + g), pack_bf16x2(o[8 * g] * inv, o[8 * g + 1] * inv),
                 pack_bf16x2(o[8 * g + 2] * inv, o[8 * g + 3] * inv), pack_bf16x2(o[8 * g + 4] * inv, o[8 * g + 5] * inv),
                 pack_bf16x2(o[8 * g + 6] * inv, o[8 * g + 7] * inv));
      }
      lse[static_cast<long long>(n) * s + qb * kRows + row] = (m + log2f(l)) * kLn2;
      fence_async_smem();
    }
    softmax_sync();
    if (ok && threadIdx.x == kSoftmax0 * 32) {
      tma_store_2d(&maps.o, sQ, col0, row0);
      tma_store_2d(&maps.o, sQ + kHalf, col0 + 64, row0);
      bulk_commit();
      bulk_wait_all();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace flash

bool attn_flash_fwd_supported(int dh) { return dh == flash::kDh; }

cudaError_t launch_attn_flash_fwd(const bf16* q, const bf16* k, const bf16* v, bf16* o, int b, int s, int H, int dh,
                                  float scale, float* lse, unsigned* err, cudaStream_t st) {
  using namespace flash;
  if (dh != kDh || s % kRows) return cudaErrorInvalidValue;
  Maps maps;
  memset(&maps, 0, sizeof(maps));
  const long long cols = 1LL * H * dh, rows = 1LL * b * s;
  bool ok = umma::encode_operand(&maps.q, q, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.k, k, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.v, v, cols, rows, cols, 64, 64) &&
            umma::encode_operand(&maps.o, o, cols, rows, cols, 64, kRows);
  if (!ok) return cudaErrorInvalidValue;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 32) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(attn_flash_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  const long long blocks = 1LL * b * H * (s / kRows);
  if (blocks == 0) return cudaSuccess;
  return launch_pdl(attn_flash_fwd_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), kSmem, st, maps,
                    b * H, H, s, scale, lse, err);
}

}  // namespace lr
