// Causal attention backward without materialised P (tcgen05, dh = 128): dK, dV and the scaled dS of
// every head in one persistent launch; dQ = dS K follows as one GEMM over the stored dS^T.
//
// A work item is a block of 128 keys j of one head (taken from a global counter, in groups of heads whose
// Q and dO fit in L2, the blocks with the most queries first).  The CTA keeps K_j and V_j in shared memory
// and walks the query steps i = 64-query blocks from the diagonal on, with the keys on the MMA rows:
//
//   S^T  = K_j Q_i^T, dP^T = V_j dO_i^T        MMA, fp32 in TMEM (two buffers: step i+1 overlaps the
//                                              element-wise work of step i)
//   P^T  = 2^(c S^T - lse log2 e)              element-wise warps, c = scale log2 e (lse: the forward's
//   dS^T = scale P^T (dP^T - D)                 row log-sum-exp; D_q = sum dO_q O_q); causal mask on the
//                                              diagonal; both written back to TMEM as bf16 over the
//                                              columns they were computed from, dS^T also to memory
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i         MMA with A from TMEM, fp32 accumulators in TMEM
//
// and at the end of the item dV_j and dK_j go to the token-major outputs.  The stored dS^T is head-major
// [b*H*s keys, s queries]; entries above the diagonal are not written except for key block j against
// query block j - 1 when j is odd, which are zeroed: the dQ GEMM's causal K range of a 256-query tile ends
// at its last query, so it reads that block.
//
// Warps: 0 item scheduler and TMA producer (K_j, V_j per item; Q_i, dO_i, lse_i, D_i per step into a
// four-stage ring), 1 TMEM allocator and MMA issuer (one lane), 2-3 idle, 4-11 element-wise: warp w reads
// TMEM lanes 32 (w mod 4) .. (its 32 keys), warpgroup 0 queries 0-31 of each step, warpgroup 1 queries
// 32-63.  TMEM: buffer b of S^T at columns 128 b, of dP^T at 128 b + 64 (64 columns each), dV at 256, dK
// at 384.  Every mbarrier wait is bounded (error word, abort flag; each role drains what it issued).
#include "attn_flash.cuh"
#include "attn_kernels.cuh"

namespace lr {
namespace flash {
namespace bwd {

constexpr int kQ = 64;                // queries per step (N of the S^T and dP^T MMAs)
constexpr int kQTile = kQ * kDh * 2;  // 16 KB: 64 rows x 128 bf16
constexpr int kQHalf = kQTile / 2;    // 8 KB: 64 rows x 64 columns
constexpr int kStages = 4;
constexpr int kSmem = 1024 + 2 * kTile + kStages * 2 * kQTile + kStages * 2 * kQ * 4 + 256;

struct Maps {
  CUtensorMap q, dout, k, v;  // q, dout: boxes of 64 columns x 64 rows; k, v: 64 x 128
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void stg_zero64(bf16* p) {  // 64 bytes of zeros (16-byte aligned)
  uint4* q = reinterpret_cast<uint4*>(p);
#pragma unroll
  for (int u = 0; u < 4; ++u) q[u] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_flash_bwd_kernel(const __grid_constant__ Maps maps, const float* lse, const float* Dr, bf16* dst, bf16* dk,
                          bf16* dv, int nheads, int H, int s, int group, float scale, unsigned* sched, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTile;
  uint8_t* sQ = sV + kTile;                // [kStages]
  uint8_t* sdO = sQ + kStages * kQTile;    // [kStages]
  float* sL = reinterpret_cast<float*>(sdO + kStages * kQTile);  // [kStages][kQ] lse
  float* sD = sL + kStages * kQ;                                   // [kStages][kQ] D
  uint64_t* bars = reinterpret_cast<uint64_t*>(sD + kStages * kQ);
  uint64_t* kv_full = bars;
  uint64_t* kv_free = bars + 1;     // the item's last S^T and dP^T MMAs have read K and V
  uint64_t* qd_full = bars + 2;     // [kStages]
  uint64_t* qd_empty = bars + 6;    // [kStages] the step's dV and dK MMAs have read Q and dO
  uint64_t* s_full = bars + 10;     // [2]
  uint64_t* p_full = bars + 12;     // [2]
  uint64_t* acc_full = bars + 14;   // the item's last dV and dK MMAs are complete
  uint64_t* acc_free = bars + 15;   // the element-wise warps have read dV and dK
  uint64_t* drain = bars + 16;
  uint64_t* item_full = bars + 17;  // [2] the item ring
  uint64_t* item_empty = bars + 19; // [2]
  int* sitem = reinterpret_cast<int*>(bars + 21);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sitem + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = s / kRows, nqs = s / kQ;
  const int items = nheads * nkb;
  constexpr int kItemReaders = 1 + 8;  // MMA issuer, element-wise warps

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_free, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kItemReaders);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_free, 8);
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

  auto next_item = [&](int k, int& t) -> bool {
    const int slot = k & 1;
    if (!mbar_wait(&item_full[slot], static_cast<uint32_t>((k >> 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA))
      return false;
    t = *reinterpret_cast<volatile int*>(&sitem[slot]);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ scheduler and TMA producer
      bool ok = true;
      int kv_issued = 0;
      long long g = 0;  // query steps issued over all items
      for (int it = 0;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&item_empty[slot], static_cast<uint32_t>((it >> 1) & 1) ^ 1u, abort_flag, err,
                       DEV_ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        const unsigned tk = atomicAdd(sched, 1u);
        const int t = tk < static_cast<unsigned>(items) ? static_cast<int>(tk) : -1;
        sitem[slot] = t;
        mbar_arrive(&item_full[slot]);
        if (t < 0) break;
        int j, n;
        item_of(t, nheads, nkb, group, j, n);  // rank 0: key block 0 (the most query steps)
        const int bi = n / H, h = n - bi * H;
        const int col0 = h * kDh;
        if (!mbar_wait(kv_free, static_cast<uint32_t>(it & 1) ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        mbar_expect_tx(kv_full, 2 * kTile);
        const int key0 = bi * s + j * kRows;
        tma_load_2d(sK, &maps.k, kv_full, col0, key0);
        tma_load_2d(sK + kHalf, &maps.k, kv_full, col0 + 64, key0);
        tma_load_2d(sV, &maps.v, kv_full, col0, key0);
        tma_load_2d(sV + kHalf, &maps.v, kv_full, col0 + 64, key0);
        ++kv_issued;
        for (int i = 2 * j; i < nqs && ok; ++i, ++g) {
          const int st = static_cast<int>(g & (kStages - 1));
          const uint32_t ph = static_cast<uint32_t>((g / kStages) & 1);
          if (!mbar_wait(&qd_empty[st], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&qd_full[st], 2 * kQTile + 2 * kQ * 4);
          const int row = bi * s + i * kQ;
          tma_load_2d(sQ + st * kQTile, &maps.q, &qd_full[st], col0, row);
          tma_load_2d(sQ + st * kQTile + kQHalf, &maps.q, &qd_full[st], col0 + 64, row);
          tma_load_2d(sdO + st * kQTile, &maps.dout, &qd_full[st], col0, row);
          tma_load_2d(sdO + st * kQTile + kQHalf, &maps.dout, &qd_full[st], col0 + 64, row);
          const long long r0 = 1LL * n * s + 1LL * i * kQ;  // head-major row of lse and D
          bulk_load(sL + st * kQ, lse + r0, kQ * 4, &qd_full[st]);
          bulk_load(sD + st * kQ, Dr + r0, kQ * 4, &qd_full[st]);
        }
        if (!ok) break;
      }
      if (!ok) {  // wait (bounded) for the copies still in flight before the CTA may exit
        for (long long k = (g > kStages ? g - kStages : 0); k < g; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(&qd_full[k & (kStages - 1)], static_cast<uint32_t>((k / kStages) & 1)) &&
                 global_timer_ns() - t0 < umma::kWaitLimitNs) {
          }
        }
        const uint64_t t0 = global_timer_ns();
        while (kv_issued > 0 && !mbar_test(kv_full, static_cast<uint32_t>((kv_issued - 1) & 1)) &&
               global_timer_ns() - t0 < umma::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS = idesc_m128<false, kQ>();  // S^T, dP^T: keys x 64 queries, both K-major
      constexpr uint32_t kIdG = idesc_m128<true, kDh>();  // dV, dK: A from TMEM, B (dO, Q) MN-major
      const uint32_t k_base = smem_addr(sK), v_base = smem_addr(sV);
      const uint32_t q_base = smem_addr(sQ), do_base = smem_addr(sdO);
      bool ok = true;
      long long g = 0;
      // S^T and dP^T of step gg into TMEM buffer gg & 1 (last held the P^T and dS^T of step gg - 2, whose
      // dV and dK MMAs were issued before this: the MMAs of a thread run in order).
      auto issue_s = [&](long long gg, bool last) -> bool {
        const int st = static_cast<int>(gg & (kStages - 1));
        const uint32_t ph = static_cast<uint32_t>((gg / kStages) & 1);
        if (!mbar_wait(&qd_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) return false;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(gg & 1) * 128;
        const uint32_t qt = q_base + st * kQTile, dt = do_base + st * kQTile;
#pragma unroll
        for (int kk = 0; kk < kDh / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * kHalf + (kk & 3) * 32, bo = (kk >> 2) * kQHalf + (kk & 3) * 32;
          mma1(d, sdesc(k_base + ao, 16, 1024), sdesc(qt + bo, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < kDh / 16; ++kk) {
          const uint32_t ao = (kk >> 2) * kHalf + (kk & 3) * 32, bo = (kk >> 2) * kQHalf + (kk & 3) * 32;
          mma1(d + 64, sdesc(v_base + ao, 16, 1024), sdesc(dt + bo, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        commit1(&s_full[gg & 1]);
        if (last) commit1(kv_free);  // K and V may be replaced once these are complete
        return true;
      };
      for (int it = 0; ok; ++it) {
        int t;
        if (!next_item(it, t)) {
          ok = false;
          break;
        }
        mbar_arrive(&item_empty[it & 1]);
        if (t < 0) break;
        int j, n;
        item_of(t, nheads, nkb, group, j, n);
        const int nsteps = nqs - 2 * j;
        if (!mbar_wait(kv_full, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA) ||
            !issue_s(g, nsteps == 1)) {
          ok = false;
          break;
        }
        for (int k = 0; k < nsteps && ok; ++k, ++g) {
          if (k + 1 < nsteps && !issue_s(g + 1, k + 2 == nsteps)) {
            ok = false;
            break;
          }
          const int b = static_cast<int>(g & 1);
          const int st = static_cast<int>(g & (kStages - 1));
          if (!mbar_wait(&p_full[b], static_cast<uint32_t>((g >> 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          // The item's first dV / dK MMAs overwrite the accumulators: the previous item's must have been read.
          if (k == 0 && !mbar_wait(acc_free, static_cast<uint32_t>(it & 1) ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qt = q_base + st * kQTile, dt = do_base + st * kQTile;
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk) {
            // K step kk = queries 16 kk .. 16 kk + 15: packed in columns 32 (kk / 2) + 8 (kk mod 2) of the
            // buffer (each warpgroup wrote its 32 queries over the first half of the columns it read)
            const uint32_t pc = static_cast<uint32_t>(b) * 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
            mma1_ta(tmem + 256, tmem + pc, sdesc(dt + kk * 2048, kQHalf, 1024), kIdG, acc);
            mma1_ta(tmem + 384, tmem + pc + 64, sdesc(qt + kk * 2048, kQHalf, 1024), kIdG, acc);
          }
          commit1(&qd_empty[st]);
          if (k + 1 == nsteps) commit1(acc_full);
        }
      }
      commit1(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_test(drain, 0) && global_timer_ns() - t0 < umma::kWaitLimitNs) {
      }
    }
  } else if (warp >= kSoftmax0) {
    // ------------------------------------------------ element-wise warps
    // `fail`: a wait of this warp gave up (its TMEM accesses and stores are skipped from then on); `ok`
    // changes only at softmax_sync_and, so every warp leaves the item loop at the same barrier.
    const int q4 = warp & 3;
    const int half = (warp - kSoftmax0) >> 2;  // queries 32 half .. 32 half + 31 of each step
    const int row = q4 * 32 + lane;            // key within the block (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float c = scale * kLog2e;
    const int HD = H * kDh;
    bool ok = true, fail = false;
    long long g = 0;
    for (int it = 0;; ++it) {
      int t = -1;
      bool okw = next_item(it, t);
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[it & 1]);
      ok = softmax_sync_and(okw && !fail);
      if (!ok || t < 0) break;
      int j, n;
      item_of(t, nheads, nkb, group, j, n);
      const int bi = n / H, h = n - bi * H;
      const int nsteps = nqs - 2 * j;
      bf16* ds_row = dst + (1LL * n * s + 1LL * j * kRows + row) * s;  // this key's row of dS^T
      if (j & 1) stg_zero64(ds_row + (j - 1) * kRows + 64 * half), stg_zero64(ds_row + (j - 1) * kRows + 64 * half + 32);
      for (int k = 0; k < nsteps; ++k, ++g) {
        const int b = static_cast<int>(g & 1);
        const int st = static_cast<int>(g & (kStages - 1));
        okw = mbar_wait(&s_full[b], static_cast<uint32_t>((g >> 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE) &&
              mbar_wait(&qd_full[st], static_cast<uint32_t>((g / kStages) & 1), abort_flag, err,
                        DEV_ERR_TIMEOUT_EPILOGUE);  // complete already; orders the reads of lse and D
        okw = __all_sync(0xffffffffu, okw);
        fail = fail || !okw;
        float x[32], y[32];
        if (!fail) {
          tc_fence_after();
          tmem_ld32(t_lane + b * 128 + 32 * half, x);
          tmem_ld32(t_lane + b * 128 + 64 + 32 * half, y);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) x[u] = y[u] = 0.f;
        }
        const float* Ls = sL + st * kQ + 32 * half;
        const float* Ds = sD + st * kQ + 32 * half;
        const int qrel = 64 * k + 32 * half - row;  // query - key of column 0 (relative to the block)
        uint32_t pk[16], dk2[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          float p[2], d2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float pe = ex2_ftz(fmaf(x[u + e], c, -Ls[u + e] * kLog2e));
            if (qrel + u + e < 0) pe = 0.f;  // a query before this key (only on the diagonal steps)
            p[e] = pe;
            d2[e] = scale * pe * (y[u + e] - Ds[u + e]);
          }
          pk[u >> 1] = pack_bf16x2(p[0], p[1]);
          dk2[u >> 1] = pack_bf16x2(d2[0], d2[1]);
        }
        if (!fail) {
          tmem_st16u(t_lane + b * 128 + 32 * half, pk);
          tmem_st16u(t_lane + b * 128 + 64 + 32 * half, dk2);
          uint4* o = reinterpret_cast<uint4*>(ds_row + (2 * j + k) * kQ + 32 * half);
#pragma unroll
          for (int u = 0; u < 4; ++u) o[u] = make_uint4(dk2[4 * u], dk2[4 * u + 1], dk2[4 * u + 2], dk2[4 * u + 3]);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[b]);
      }
      // dV_j and dK_j: this warp's 32 keys, dh columns 64 half .. 64 half + 63
      okw = mbar_wait(acc_full, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
      okw = __all_sync(0xffffffffu, okw);
      fail = fail || !okw;
      if (!fail) {
        tc_fence_after();
        const long long orow = (1LL * bi * s + 1LL * j * kRows + row) * HD + 1LL * h * kDh + 64 * half;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          bf16* out = (which == 0 ? dv : dk) + orow;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float a[32];
            tmem_ld32(t_lane + 256 + 128 * which + 64 * half + 32 * cc, a);
            tmem_ld_wait();
            uint4* o = reinterpret_cast<uint4*>(out + 32 * cc);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              o[u] = make_uint4(pack_bf16x2(a[8 * u], a[8 * u + 1]), pack_bf16x2(a[8 * u + 2], a[8 * u + 3]),
                                pack_bf16x2(a[8 * u + 4], a[8 * u + 5]), pack_bf16x2(a[8 * u + 6], a[8 * u + 7]));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

}  // namespace bwd
}  // namespace flash

cudaError_t launch_attn_flash_bwd(const bf16* q, const bf16* k, const bf16* v, const bf16* dout, const float* lse,
                                  const float* D, bf16* dst, bf16* dk, bf16* dv, int b, int s, int H, int dh,
                                  float scale, unsigned* sched, unsigned* err, cudaStream_t st) {
  using namespace flash;
  using namespace flash::bwd;
  if (dh != kDh || s % kRows) return cudaErrorInvalidValue;
  bwd::Maps maps;
  memset(&maps, 0, sizeof(maps));
  const long long cols = 1LL * H * dh, rows = 1LL * b * s;
  bool ok = umma::encode_operand(&maps.q, q, cols, rows, cols, 64, kQ) &&
            umma::encode_operand(&maps.dout, dout, cols, rows, cols, 64, kQ) &&
            umma::encode_operand(&maps.k, k, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.v, v, cols, rows, cols, 64, kRows);
  if (!ok) return cudaErrorInvalidValue;
  static int configured_mask = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 32) return cudaErrorInvalidDevice;
  if (!(__atomic_load_n(&configured_mask, __ATOMIC_ACQUIRE) & (1 << dev))) {
    cudaError_t e = cudaFuncSetAttribute(attn_flash_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    __atomic_fetch_or(&configured_mask, 1 << dev, __ATOMIC_RELEASE);
  }
  const long long items = 1LL * b * H * (s / kRows);
  if (items == 0) return cudaSuccess;
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  const int group = heads_per_group(1LL * b * H, 4LL * s * dh);  // Q and dO of a head: s x dh x 2 x 2 bytes
  cudaError_t e = cudaMemsetAsync(sched, 0, sizeof(unsigned), st);  // the item counter of this launch
  if (e != cudaSuccess) return e;
  const long long grid = std::min<long long>(items, device_sm_count());
  return launch_pdl(attn_flash_bwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmem, st, maps, lse,
                    D, dst, dk, dv, b * H, H, s, group, scale, sched, err);
}

}  // namespace lr
