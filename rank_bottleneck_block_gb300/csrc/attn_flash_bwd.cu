// Causal attention backward without materialised P (tcgen05, dh = 128): dK, dV and the scaled dS of
// every head in one persistent launch; dQ = dS K follows as one GEMM over the stored dS^T.
//
// A work item is a block of 128 keys j of one head (taken from a global counter, in groups of heads whose
// Q and dO fit in L2, the blocks with the most queries first).  The CTA keeps K_j and V_j in shared memory
// and walks the query blocks i = j, j+1, ... of 128 queries, with the keys on the MMA rows:
//
//   S^T  = K_j Q_i^T, dP^T = V_j dO_i^T        MMA (N = 128), fp32 in TMEM
//   P^T  = 2^(c S^T - lse log2 e)              element-wise warps, c = scale log2 e (lse: the forward's
//   dS^T = scale P^T (dP^T - D)                 row log-sum-exp; D_q = sum dO_q O_q); causal mask on the
//                                              diagonal block; both written back to TMEM as bf16 over the
//                                              columns they were computed from, dS^T also to memory
//   dV_j += P^T dO_i,  dK_j += dS^T Q_i         MMA with A from TMEM, fp32 accumulators in TMEM
//
// TMEM holds S^T, dP^T, dV and dK (128 columns each), so S^T and dP^T have one buffer.  The element-wise
// warps work on the block's queries in two halves of 64, and the dV and dK MMAs of the first half run
// while they compute the second.  At the end of the item dV_j and dK_j go to the token-major outputs.
// The stored dS^T is head-major [b*H*s keys, s queries]; entries above the diagonal are not written
// except for key block j against query block j - 1 when j is odd, which are zeroed: the dQ GEMM's causal
// K range of a 256-query tile ends at its last query, so it reads that block.
//
// Warps: 0 item scheduler and TMA producer (K_j, V_j per item; Q_i, dO_i, lse_i, D_i per query block
// into a two-stage ring), 1 TMEM allocator and MMA issuer (one lane), 2-3 idle, 4-19 element-wise: warp w
// reads TMEM lanes 32 (w mod 4) .. (its 32 keys) and takes queries 64 h + 16 sub .. + 15 of half h
// (sub = (w - 4) / 4); each warp writes its 32 x 16 pieces of dS^T, dK and dV through its own staging
// tile with TMA stores.  TMEM: S^T at columns 0, dP^T at 128, dV at 256, dK at 384.  Every mbarrier wait
// is bounded (error word, abort flag; each role drains what it issued).
#include "attn_flash.cuh"
#include "attn_kernels.cuh"

namespace lr {
namespace flash {
namespace bwd {

constexpr int kQ = kRows;             // queries per step (N of the S^T and dP^T MMAs)
constexpr int kQTile = kTile;         // 32 KB: 128 rows x 128 bf16
constexpr int kStages = 2;
constexpr int kEw = 16;                          // element-wise warps (4 per TMEM lane quarter)
constexpr int kThreadsB = 32 * (kSoftmax0 + kEw);  // 640
constexpr int kStageDs = 32 * 16 * 2;  // one warp's 32 rows x 16 columns, staged for a TMA store (1 KB)
constexpr int kSmem = 1024 + 2 * kTile + kStages * 2 * kQTile + kEw * kStageDs + kStages * 2 * kQ * 4 + 256;

using umma::tmem_ld16;

struct Maps {
  CUtensorMap q, dout, k, v;  // boxes of 64 columns x 128 rows
  CUtensorMap ds, dk, dv;     // outputs: boxes of 16 columns x 32 rows, 32-byte swizzle
};

// 32 lanes x 8 consecutive 32-bit columns from registers.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// The sixteen element-wise warps' named barrier, returning the AND of `ok` over them.
__device__ __forceinline__ bool ew_sync_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, 1, 512, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

// Byte offset of 16-byte chunk u of row r in a staging tile of 32-byte rows with the 32-byte swizzle.
__device__ __forceinline__ uint32_t sw32_off(int r, int u) { return r * 32 + ((u ^ ((r >> 2) & 1)) << 4); }

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

// P^T and scale dS^T of 16 queries of one key row (the element-wise step), packed in bf16 pairs.
template <bool MASK>
__device__ __forceinline__ void pds16(const float* x, const float* y, const float* Ls, const float* Ds, float c,
                                      float scale, int qrel, uint32_t* pk, uint32_t* dk2) {
#pragma unroll
  for (int u4 = 0; u4 < 4; ++u4) {
    const float4 l4 = *reinterpret_cast<const float4*>(Ls + 4 * u4);
    const float4 d4 = *reinterpret_cast<const float4*>(Ds + 4 * u4);
    const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
    float p[4], d2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int u = 4 * u4 + e;
      float pe = ex2_ftz(fmaf(x[u], c, -lv[e] * kLog2e));
      if (MASK && qrel + u < 0) pe = 0.f;  // a query before this key (the diagonal block)
      p[e] = pe;
      d2[e] = scale * pe * (y[u] - dv[e]);
    }
    pk[2 * u4] = pack_bf16x2(p[0], p[1]);
    pk[2 * u4 + 1] = pack_bf16x2(p[2], p[3]);
    dk2[2 * u4] = pack_bf16x2(d2[0], d2[1]);
    dk2[2 * u4 + 1] = pack_bf16x2(d2[2], d2[3]);
  }
}

__global__ void __launch_bounds__(kThreadsB, 1)
    attn_flash_bwd_kernel(const __grid_constant__ Maps maps, const float* lse, const float* Dr, bf16* dst, bf16* dk,
                          bf16* dv, int nheads, int H, int s, int group, float scale, unsigned* sched, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem;
  uint8_t* sV = sK + kTile;
  uint8_t* sQ = sV + kTile;              // [kStages]
  uint8_t* sdO = sQ + kStages * kQTile;  // [kStages]
  uint8_t* sS = sdO + kStages * kQTile;  // [kEw] output staging, one tile per element-wise warp
  float* sL = reinterpret_cast<float*>(sS + kEw * kStageDs);  // [kStages][kQ] lse
  float* sD = sL + kStages * kQ;                                   // [kStages][kQ] D
  uint64_t* bars = reinterpret_cast<uint64_t*>(sD + kStages * kQ);
  uint64_t* kv_full = bars;
  uint64_t* kv_free = bars + 1;     // the item's last S^T and dP^T MMAs have read K and V
  uint64_t* qd_full = bars + 2;     // [kStages]
  uint64_t* qd_empty = bars + 4;    // [kStages] the step's dV and dK MMAs have read Q and dO
  uint64_t* s_full = bars + 6;      // S^T and dP^T of the step are in TMEM
  uint64_t* p_half = bars + 7;      // [2] P^T and dS^T of a half of the step's queries are in TMEM
  uint64_t* acc_full = bars + 9;    // the item's last dV and dK MMAs are complete
  uint64_t* acc_free = bars + 10;   // the element-wise warps have read dV and dK
  uint64_t* drain = bars + 11;
  uint64_t* item_full = bars + 12;  // [2] the item ring
  uint64_t* item_empty = bars + 14; // [2]
  int* sitem = reinterpret_cast<int*>(bars + 16);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sitem + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nkb = s / kRows;
  const int items = nheads * nkb;
  constexpr int kItemReaders = 1 + kEw;  // MMA issuer, element-wise warps

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(kv_free, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&qd_full[i], 1);
      mbar_init(&qd_empty[i], 1);
    }
    mbar_init(s_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_half[i], kEw);
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kItemReaders);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_free, kEw);
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
      long long g = 0;  // query blocks issued over all items
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
        item_of(t, nheads, nkb, group, j, n);  // rank 0: key block 0 (the most query blocks)
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
        for (int i = j; i < nkb && ok; ++i, ++g) {
          const int st = static_cast<int>(g & 1);
          const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
          if (!mbar_wait(&qd_empty[st], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&qd_full[st], 2 * kQTile + 2 * kQ * 4);
          const int row = bi * s + i * kQ;
          tma_load_2d(sQ + st * kQTile, &maps.q, &qd_full[st], col0, row);
          tma_load_2d(sQ + st * kQTile + kHalf, &maps.q, &qd_full[st], col0 + 64, row);
          tma_load_2d(sdO + st * kQTile, &maps.dout, &qd_full[st], col0, row);
          tma_load_2d(sdO + st * kQTile + kHalf, &maps.dout, &qd_full[st], col0 + 64, row);
          const long long r0 = 1LL * n * s + 1LL * i * kQ;  // head-major row of lse and D
          bulk_load(sL + st * kQ, lse + r0, kQ * 4, &qd_full[st]);
          bulk_load(sD + st * kQ, Dr + r0, kQ * 4, &qd_full[st]);
        }
        if (!ok) break;
      }
      if (!ok) {  // wait (bounded) for the copies still in flight before the CTA may exit
        for (long long k = (g > kStages ? g - kStages : 0); k < g; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(&qd_full[k & 1], static_cast<uint32_t>((k >> 1) & 1)) &&
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
      constexpr uint32_t kIdS = idesc_m128<false, kQ>();  // S^T, dP^T: keys x 128 queries, both K-major
      constexpr uint32_t kIdG = idesc_m128<true, kDh>();  // dV, dK: A from TMEM, B (dO, Q) MN-major
      const uint32_t k_base = smem_addr(sK), v_base = smem_addr(sV);
      const uint32_t q_base = smem_addr(sQ), do_base = smem_addr(sdO);
      bool ok = true;
      long long g = 0;
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
        const int nsteps = nkb - j;
        if (!mbar_wait(kv_full, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int k = 0; k < nsteps && ok; ++k, ++g) {
          const int st = static_cast<int>(g & 1);
          if (!mbar_wait(&qd_full[st], static_cast<uint32_t>((g >> 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t qt = q_base + st * kQTile, dt = do_base + st * kQTile;
          // S^T and dP^T (their columns last held the previous step's P^T and dS^T, whose dV and dK MMAs
          // were issued before these: the MMAs of a thread run in order)
#pragma unroll
          for (int kk = 0; kk < kDh / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kHalf + (kk & 3) * 32;
            mma1(tmem, sdesc(k_base + o, 16, 1024), sdesc(qt + o, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < kDh / 16; ++kk) {
            const uint32_t o = (kk >> 2) * kHalf + (kk & 3) * 32;
            mma1(tmem + 128, sdesc(v_base + o, 16, 1024), sdesc(dt + o, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
          }
          commit1(s_full);
          if (k + 1 == nsteps) commit1(kv_free);  // K and V may be replaced once these are complete
          for (int hf = 0; hf < 2 && ok; ++hf) {
            if (!mbar_wait(&p_half[hf], static_cast<uint32_t>(g & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            // The item's first dV / dK MMAs overwrite the accumulators: the previous item's must have been read.
            if (k == 0 && hf == 0 &&
                !mbar_wait(acc_free, static_cast<uint32_t>(it & 1) ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int kq = 0; kq < 4; ++kq) {
              // K step kk = queries 16 kk .. 16 kk + 15, packed by the warps of column group kk mod 4 of half
              // kk / 4 in columns 64 (kk / 4) + 16 (kk mod 4) .. + 7: over the first half of what they read
              const int kk = 4 * hf + kq;
              const uint32_t pc = 64 * (kk >> 2) + 16 * (kk & 3);
              const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
              mma1_ta(tmem + 256, tmem + pc, sdesc(dt + kk * 2048, kHalf, 1024), kIdG, acc);
              mma1_ta(tmem + 384, tmem + 128 + pc, sdesc(qt + kk * 2048, kHalf, 1024), kIdG, acc);
            }
          }
          if (!ok) break;
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
    // changes only at ew_sync_and, so every warp leaves the item loop at the same barrier.
    const int q4 = warp & 3;
    const int sub = (warp - kSoftmax0) >> 2;  // column group: queries 64 h + 16 sub .. + 15 of half h
    const int row = q4 * 32 + lane;           // key within the block (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const float c = scale * kLog2e;
    const uint32_t tile = smem_addr(sS + (warp - kSoftmax0) * kStageDs);
    uint8_t* tile_p = sS + (warp - kSoftmax0) * kStageDs;
    bool ok = true, fail = false;
    long long g = 0;
    // 32 rows x 16 bf16 (this warp's 8 packed words per lane) through the staging tile to a TMA store.
    auto store_tile = [&](const CUtensorMap* map, const uint32_t* w, int x, int y) {
      if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the tile is free
      __syncwarp();
      sts128(tile + sw32_off(lane, 0), w[0], w[1], w[2], w[3]);
      sts128(tile + sw32_off(lane, 1), w[4], w[5], w[6], w[7]);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_2d(map, tile_p, x, y);
        bulk_commit();
      }
    };
    for (int it = 0;; ++it) {
      int t = -1;
      bool okw = next_item(it, t);
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[it & 1]);
      ok = ew_sync_and(okw && !fail);
      if (!ok || t < 0) break;
      int j, n;
      item_of(t, nheads, nkb, group, j, n);
      const int bi = n / H, h = n - bi * H;
      const int nsteps = nkb - j;
      const int ds_key0 = n * s + j * kRows + q4 * 32;  // this warp's first key row of dS^T
      if (j & 1) stg_zero64(dst + (1LL * n * s + 1LL * j * kRows + row) * s + (j - 1) * kRows + 32 * sub);
      for (int k = 0; k < nsteps; ++k, ++g) {
        const int st = static_cast<int>(g & 1);
        okw = mbar_wait(s_full, static_cast<uint32_t>(g & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE) &&
              mbar_wait(&qd_full[st], static_cast<uint32_t>((g >> 1) & 1), abort_flag, err,
                        DEV_ERR_TIMEOUT_EPILOGUE);  // complete already; orders the reads of lse and D
        okw = __all_sync(0xffffffffu, okw);
        fail = fail || !okw;
        uint32_t dsk[2][8];  // this warp's scale dS^T of both halves, stored after the second (the warps
                             // then wait for the next step's S^T anyway)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          const int c0 = 64 * hf + 16 * sub;  // this warp's 16 queries of the block
          float x[16], y[16];
          if (!fail) {
            tc_fence_after();
            tmem_ld16(t_lane + c0, x);
            tmem_ld16(t_lane + 128 + c0, y);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int u = 0; u < 16; ++u) x[u] = y[u] = 0.f;
          }
          const float* Ls = sL + st * kQ + c0;
          const float* Ds = sD + st * kQ + c0;
          uint32_t pk[8];
          uint32_t* dk2 = dsk[hf];
          if (k == 0)
            pds16<true>(x, y, Ls, Ds, c, scale, c0 - row, pk, dk2);
          else
            pds16<false>(x, y, Ls, Ds, c, scale, 0, pk, dk2);
          if (!fail) {
            tmem_st8u(t_lane + c0, pk);
            tmem_st8u(t_lane + 128 + c0, dk2);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_half[hf]);
        }
        if (!fail) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) store_tile(&maps.ds, dsk[hf], (j + k) * kQ + 64 * hf + 16 * sub, ds_key0);
        }
      }
      // dV_j and dK_j: this warp's 32 keys, dh columns 32 sub .. 32 sub + 31 of each
      okw = mbar_wait(acc_full, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
      okw = __all_sync(0xffffffffu, okw);
      fail = fail || !okw;
      if (!fail) tc_fence_after();
#pragma unroll
      for (int which = 0; which < 2; ++which)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          float a[16];
          if (!fail) {
            tmem_ld16(t_lane + 256 + 128 * which + 32 * sub + 16 * hh, a);
            tmem_ld_wait();
          }
          if (which == 1 && hh == 1) {  // the accumulators are read; the last store below uses registers
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free);
          }
          if (!fail) {
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) w[u] = pack_bf16x2(a[2 * u], a[2 * u + 1]);
            store_tile(which == 0 ? &maps.dv : &maps.dk, w, h * kDh + 32 * sub + 16 * hh, bi * s + j * kRows + q4 * 32);
          }
        }
    }
    if (lane == 0) bulk_wait_all();  // this warp's stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// bf16 [rows, cols] row-major (ld = cols) output map: boxes of 16 columns x 32 rows, 32-byte swizzle.
inline bool encode_out16(CUtensorMap* m, const void* ptr, long long cols, long long rows) {
  const long long dims[2] = {cols, rows}, strides[1] = {cols};
  const int box[2] = {16, 32};
  return umma::encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_32B);
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
  bool ok = umma::encode_operand(&maps.q, q, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.dout, dout, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.k, k, cols, rows, cols, 64, kRows) &&
            umma::encode_operand(&maps.v, v, cols, rows, cols, 64, kRows) &&
            encode_out16(&maps.ds, dst, s, 1LL * b * H * s) && encode_out16(&maps.dk, dk, cols, rows) &&
            encode_out16(&maps.dv, dv, cols, rows);
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
  return launch_pdl(attn_flash_bwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreadsB), kSmem, st, maps, lse,
                    D, dst, dk, dv, b * H, H, s, group, scale, sched, err);
}

}  // namespace lr
