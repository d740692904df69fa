// Causal attention forward without materialised scores (tcgen05, dh = 128).
//
// A persistent grid (one CTA per SM) takes work items of 128 queries of one head (query block i) from a
// global counter, in groups of heads whose K and V fit in L2 and heaviest first inside a group; for
// each item the CTA walks the key blocks 0 .. i of 128 keys:
//
//   S_j = Q K_j^T                      MMA, fp32 in TMEM (two buffers: S_{j+1} overlaps the softmax of j)
//   P_j = 2^(c S_j - m)                the softmax warps, c = scale log2(e); m is the row's running
//                                      maximum of c S, raised lazily; P_j (bf16) is written back into
//                                      the columns of S_j's TMEM buffer
//   O  += P_j V_j                      MMA with A = P_j read from TMEM, fp32 accumulator in TMEM
//
// with the running row sum l = sum 2^(c S - m).  m is raised only when a block's maximum exceeds it by
// more than 8 (powers of two): P then stays below 2^8 and O, l keep their scale until a real change, at
// which point the row's O (TMEM) and l are multiplied by 2^(m_old - m_new) before the block's P V is
// issued.  Every formula is exact for any m; only overflow limits the laziness.  At the end O / l goes to
// the token-major output and lse = ln 2 (m + log2 l) to the head-major row log-sum-exp the backward reads.
//
// Warps: 0 item scheduler and TMA producer of Q (per item) and K_j (two-stage ring), 1 TMEM allocator and
// MMA issuer (one lane), 2 TMA producer of V_j (its own two-stage ring: K_{j+2} loads once S_j is done,
// V_{j+2} once P_j V_j is), 3 idle, 4-11 softmax and output in two warpgroups: warp w reads TMEM lanes
// 32 (w mod 4) .. (its 32 query rows); warpgroup 0 takes keys 0-63 of each block and output columns
// 0-63, warpgroup 1 keys 64-127 and columns 64-127.  The two halves of a row agree on m through shared
// memory once per block (a named barrier of the eight warps, which also orders every read of S before
// any write of P over it).  The next item's Q is loaded once the last S MMA of the current one has read
// Q, so its first S overlaps the current item's last softmax and output.  Shared memory: Q, K[2], V[2]
// and the staged output O, each 128 x 128 bf16 in the 128-byte-swizzled UMMA layouts (K-major Q, K in
// two 64-column halves; V MN-major in two 64-key halves of two 64-column chunks).  TMEM: S/P[2] at
// columns 0 and 128, O at 256.  Every mbarrier wait is bounded (error word, abort flag; each role drains
// what it issued and TMEM is freed).
#include "attn_flash.cuh"
#include "attn_kernels.cuh"

namespace lr {
namespace flash {

constexpr int kSmem = 1024 + 6 * kTile + 2048 + 256;
constexpr float kLazy = 8.f;   // raise the running maximum only past this margin (log2 domain)

struct Maps {
  CUtensorMap q, k, v, o;  // q, k, o: boxes of 64 columns x 128 rows; v: 64 x 64
};

__global__ void __launch_bounds__(kThreads, 1)
    attn_flash_fwd_kernel(const __grid_constant__ Maps maps, int nheads, int H, int s, int group, float scale,
                          float* lse, unsigned* sched, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK = sQ + kTile;      // [2]
  uint8_t* sV = sK + 2 * kTile;  // [2]
  uint8_t* sO = sV + 2 * kTile;  // the item's output, staged for the TMA store
  float* xch = reinterpret_cast<float*>(sO + kTile);  // [2 parities][2 halves][128 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(xch + 2 * 2 * kRows);
  uint64_t* q_full = bars;
  uint64_t* q_free = bars + 1;      // the item's last S MMA has read the Q tile
  uint64_t* k_full = bars + 2;      // [2]
  uint64_t* k_empty = bars + 4;     // [2] the S MMA has read K
  uint64_t* v_full = bars + 6;      // [2]
  uint64_t* v_empty = bars + 8;     // [2] the P V MMA has read V
  uint64_t* s_full = bars + 10;     // [2]
  uint64_t* p_full = bars + 12;     // [2]
  uint64_t* o_done = bars + 14;     // one completion per P V
  uint64_t* o_last = bars + 15;     // one completion per item: its last P V
  uint64_t* o_free = bars + 16;     // the softmax warps have read the item's O
  uint64_t* drain = bars + 17;
  uint64_t* item_full = bars + 18;  // [2] the item ring
  uint64_t* item_empty = bars + 20; // [2]
  int* sitem = reinterpret_cast<int*>(bars + 22);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sitem + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nqb = s / kRows;
  const int items = nheads * nqb;
  constexpr int kItemReaders = 1 + 1 + 8;  // V producer, MMA issuer, softmax warps

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);
      mbar_init(&item_full[i], 1);
      mbar_init(&item_empty[i], kItemReaders);
    }
    mbar_init(o_done, 1);
    mbar_init(o_last, 1);
    mbar_init(o_free, 8);
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

  // The k-th item of this CTA (the first negative one ends the walk), read from the ring; false when the
  // wait gave up.
  auto next_item = [&](int k, int& t) -> bool {
    const int slot = k & 1;
    if (!mbar_wait(&item_full[slot], static_cast<uint32_t>((k >> 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA))
      return false;
    t = *reinterpret_cast<volatile int*>(&sitem[slot]);
    return true;
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ scheduler and Q / K producer
      bool ok = true;
      int it = 0, q_issued = 0;
      long long g = 0;  // key blocks issued over all items
      for (;; ++it) {
        const int slot = it & 1;
        if (!mbar_wait(&item_empty[slot], static_cast<uint32_t>((it >> 1) & 1) ^ 1u, abort_flag, err,
                       DEV_ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        const unsigned tk = atomicAdd(sched, 1u);
        const int t = tk < static_cast<unsigned>(items) ? static_cast<int>(tk) : -1;
        sitem[slot] = t;
        mbar_arrive(&item_full[slot]);  // release: the item id is visible to the readers
        if (t < 0) break;
        int qb, n;
        item_of(t, nheads, nqb, group, qb, n);
        qb = nqb - 1 - qb;  // rank 0: the last query block (the most key blocks)
        const int bi = n / H, h = n - bi * H;
        const int col0 = h * kDh;
        // Q of this item once the previous item's last S MMA has read the previous Q.
        if (!mbar_wait(q_free, static_cast<uint32_t>(it & 1) ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
          ok = false;
          break;
        }
        mbar_expect_tx(q_full, kTile);
        tma_load_2d(sQ, &maps.q, q_full, col0, bi * s + qb * kRows);
        tma_load_2d(sQ + kHalf, &maps.q, q_full, col0 + 64, bi * s + qb * kRows);
        ++q_issued;
        for (int j = 0; j <= qb && ok; ++j, ++g) {
          const int st = static_cast<int>(g & 1);
          const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
          if (!mbar_wait(&k_empty[st], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&k_full[st], kTile);
          const int key0 = bi * s + j * kRows;
          tma_load_2d(sK + st * kTile, &maps.k, &k_full[st], col0, key0);
          tma_load_2d(sK + st * kTile + kHalf, &maps.k, &k_full[st], col0 + 64, key0);
        }
        if (!ok) break;
      }
      if (!ok) {  // wait (bounded) for the copies still in flight before the CTA may exit
        for (long long k = (g > 2 ? g - 2 : 0); k < g; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(&k_full[k & 1], static_cast<uint32_t>((k >> 1) & 1)) &&
                 global_timer_ns() - t0 < umma::kWaitLimitNs) {
          }
        }
        const uint64_t t0 = global_timer_ns();
        while (q_issued > 0 && !mbar_test(q_full, static_cast<uint32_t>((q_issued - 1) & 1)) &&
               global_timer_ns() - t0 < umma::kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 2) {
    if (lane == 0) {
      // ------------------------------------------------ V producer
      bool ok = true;
      long long g = 0;
      for (int it = 0;; ++it) {
        int t;
        if (!next_item(it, t)) {
          ok = false;
          break;
        }
        mbar_arrive(&item_empty[it & 1]);
        if (t < 0) break;
        int qb, n;
        item_of(t, nheads, nqb, group, qb, n);
        qb = nqb - 1 - qb;  // rank 0: the last query block (the most key blocks)
        const int bi = n / H, h = n - bi * H;
        for (int j = 0; j <= qb && ok; ++j, ++g) {
          const int st = static_cast<int>(g & 1);
          const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
          if (!mbar_wait(&v_empty[st], ph ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&v_full[st], kTile);
          const int key0 = bi * s + j * kRows;
          uint8_t* v_dst = sV + st * kTile;
          // V as the MN-major B operand: per 64-key half, two 64-column chunks of 64 keys x 128 bytes
          for (int kh = 0; kh < 2; ++kh)
            for (int ch = 0; ch < 2; ++ch)
              tma_load_2d(v_dst + kh * kHalf + ch * (kHalf / 2), &maps.v, &v_full[st], h * kDh + 64 * ch,
                          key0 + 64 * kh);
        }
        if (!ok) break;
      }
      if (!ok) {
        for (long long k = (g > 2 ? g - 2 : 0); k < g; ++k) {
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(&v_full[k & 1], static_cast<uint32_t>((k >> 1) & 1)) &&
                 global_timer_ns() - t0 < umma::kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      constexpr uint32_t kIdS = idesc_m128<false>();  // S = Q K^T: both K-major
      constexpr uint32_t kIdO = idesc_m128<true>();   // O += P V: P from TMEM, V MN-major
      const uint32_t q_base = smem_addr(sQ), k_base = smem_addr(sK), v_base = smem_addr(sV);
      bool ok = true;
      long long g = 0;  // key blocks over all items
      auto issue_s = [&](long long gg, bool last) -> bool {
        const int st = static_cast<int>(gg & 1);
        const uint32_t ph = static_cast<uint32_t>((gg >> 1) & 1);
        if (!mbar_wait(&k_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) return false;
        tc_fence_after();
        const uint32_t kt = k_base + st * kTile;
        // buffer st last held P_{gg-2}, whose P V was issued before this (the MMAs of a thread run in order)
#pragma unroll
        for (int kk = 0; kk < kDh / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma1(tmem + st * kRows, sdesc(q_base + off, 16, 1024), sdesc(kt + off, 16, 1024), kIdS, kk > 0 ? 1u : 0u);
        }
        commit1(&s_full[st]);
        commit1(&k_empty[st]);
        if (last) commit1(q_free);  // Q may be replaced once this S is complete
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
        int qb, n;
        item_of(t, nheads, nqb, group, qb, n);
        qb = nqb - 1 - qb;  // rank 0: the last query block (the most key blocks)
        if (!mbar_wait(q_full, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_MMA) ||
            !issue_s(g, qb == 0)) {
          ok = false;
          break;
        }
        for (int j = 0; j <= qb && ok; ++j, ++g) {
          if (j + 1 <= qb && !issue_s(g + 1, j + 1 == qb)) {
            ok = false;
            break;
          }
          const int st = static_cast<int>(g & 1);
          const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
          if (!mbar_wait(&p_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA) ||
              !mbar_wait(&v_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          // The item's first P V overwrites O: the previous item's O must have been read.
          if (j == 0 && !mbar_wait(o_free, static_cast<uint32_t>(it & 1) ^ 1u, abort_flag, err, DEV_ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vt = v_base + st * kTile;
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk) {  // K = the block's 128 keys: 8 packed columns each
            const uint64_t bd = sdesc(vt + (kk >> 2) * kHalf + (kk & 3) * 2048, kHalf / 2, 1024);
            mma1_ta(tmem + 2 * kRows, tmem + st * kRows + kk * 8, bd, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          }
          commit1(o_done);
          if (j == qb) commit1(o_last);
          commit1(&v_empty[st]);
        }
      }
      // Drain: every MMA issued by this thread has completed once this barrier flips.
      commit1(drain);
      const uint64_t t0 = global_timer_ns();
      while (!mbar_test(drain, 0) && global_timer_ns() - t0 < umma::kWaitLimitNs) {
      }
    }
  } else if (warp >= kSoftmax0) {
    // ------------------------------------------------ softmax and output
    // Errors: `fail` is this warp's view (a wait of its own gave up); `ok` changes only at a
    // softmax_sync_and, so it is the same in all eight warps and every branch on it that skips a named
    // barrier is taken by all of them.  A warp that failed skips its TMEM accesses and carries on to the
    // next such barrier (the abort flag makes every later wait return at once).
    const int q = warp & 3;
    const int half = (warp - kSoftmax0) >> 2;  // keys / output columns 64 half .. 64 half + 63
    const int row = q * 32 + lane;             // query row within the block (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool storer = threadIdx.x == kSoftmax0 * 32;
    const float c = scale * kLog2e;
    bool ok = true, fail = false;
    long long g = 0;
    for (int it = 0;; ++it) {
      int t = -1;
      bool okw = next_item(it, t);
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[it & 1]);
      ok = softmax_sync_and(okw && !fail);
      if (!ok || t < 0) break;  // uniform: every warp read the same item
      int qb, n;
      item_of(t, nheads, nqb, group, qb, n);
      qb = nqb - 1 - qb;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j <= qb; ++j, ++g) {
        const int st = static_cast<int>(g & 1);
        const uint32_t ph = static_cast<uint32_t>((g >> 1) & 1);
        okw = mbar_wait(&s_full[st], ph, abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
        okw = __all_sync(0xffffffffu, okw && !fail);
        float x[64];
        if (okw) {
          tc_fence_after();
          tmem_ld32(t_lane + st * kRows + 64 * half, x);
          tmem_ld32(t_lane + st * kRows + 64 * half + 32, x + 32);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int kk = 0; kk < 64; ++kk) x[kk] = 0.f;
        }
        if (j == qb) {  // the diagonal block: keys after the row's query are masked
#pragma unroll
          for (int kk = 0; kk < 64; ++kk)
            if (64 * half + kk > row) x[kk] = -INFINITY;
        }
        // Block maximum of c S (c > 0, so the maximum of S scaled), in eight independent chains.
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = x[u];
#pragma unroll
        for (int kk = 8; kk < 64; ++kk) mx[kk & 7] = fmaxf(mx[kk & 7], x[kk]);
        float bm = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        bm *= c;
        // Both halves of the row agree on the block maximum (this barrier also orders every read of
        // S_j before any write of P_j over its columns).
        float* xb = xch + (g & 1) * (2 * kRows);
        xb[half * kRows + row] = bm;
        tc_fence_before();
        ok = softmax_sync_and(okw);
        if (!ok) break;
        tc_fence_after();
        bm = fmaxf(bm, xb[(1 - half) * kRows + row]);
        // Lazy maximum: raise m (and rescale O, l) only when the block's maximum passes it by kLazy.
        const bool raise = m == -INFINITY ? true : bm > m + kLazy;
        const float m_new = raise ? fmaxf(m, bm) : m;
        const float alpha = (raise && m != -INFINITY) ? exp2f(m - m_new) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // O holds the blocks before j: wait for P_{j-1} V_{j-1}, then scale this row's half of O.  (S_j
          // complete implies P_{j-2} V_{j-2} complete, so o_done is at most one phase behind here.)
          okw = mbar_wait(o_done, static_cast<uint32_t>((g - 1) & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
          fail = !__all_sync(0xffffffffu, okw);
          if (!fail) {
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              float o[32];
              const uint32_t oa = t_lane + 2 * kRows + 64 * half + 32 * cc;
              tmem_ld32(oa, o);
              tmem_ld_wait();
#pragma unroll
              for (int u = 0; u < 32; ++u) o[u] *= alpha;
              tmem_st32(oa, o);
            }
          }
        }
        l *= alpha;
        m = m_new;
        // P = 2^(c S - m) (bf16 pairs) over the first 64 columns of S's buffer: this half's 64 keys in
        // 32 columns; the row sum in four independent chains.
        uint32_t pk[32];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
        const float nm = -m;
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const float p0 = ex2_ftz(fmaf(x[2 * u], c, nm)), p1 = ex2_ftz(fmaf(x[2 * u + 1], c, nm));
          ls[u & 3] += p0 + p1;
          pk[u] = pack_bf16x2(p0, p1);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        if (!fail) tmem_st32u(t_lane + st * kRows + 32 * half, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[st]);
      }
      if (!ok) break;  // uniform: taken after a softmax_sync_and
      // O = O / l after the item's last P V (l summed over both halves of the row), staged in sO once
      // the previous item's store has read it, then stored.
      okw = mbar_wait(o_last, static_cast<uint32_t>(it & 1), abort_flag, err, DEV_ERR_TIMEOUT_EPILOGUE);
      okw = __all_sync(0xffffffffu, okw && !fail);
      if (storer) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
      float* xb = xch + (g & 1) * (2 * kRows);
      xb[half * kRows + row] = l;
      ok = softmax_sync_and(okw);
      if (!ok) break;
      const float lt = l + xb[(1 - half) * kRows + row];
      tc_fence_after();
      const float inv = 1.f / lt;
      const uint32_t ob = smem_addr(sO);
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float o[32];
        tmem_ld32(t_lane + 2 * kRows + 64 * half + 32 * cc, o);
        tmem_ld_wait();
#pragma unroll
        for (int gq = 0; gq < 4; ++gq)
          sts128(ob + kmaj_off(row, 8 * half + 4 * cc + gq), pack_bf16x2(o[8 * gq] * inv, o[8 * gq + 1] * inv),
                 pack_bf16x2(o[8 * gq + 2] * inv, o[8 * gq + 3] * inv),
                 pack_bf16x2(o[8 * gq + 4] * inv, o[8 * gq + 5] * inv),
                 pack_bf16x2(o[8 * gq + 6] * inv, o[8 * gq + 7] * inv));
      }
      if (half == 0) lse[static_cast<long long>(n) * s + qb * kRows + row] = (m + log2f(lt)) * kLn2;
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);  // this warp has read its part of O
      softmax_sync();                        // staging complete; every partner has read l
      if (storer) {
        const int bi = n / H, h = n - bi * H;
        tma_store_2d(&maps.o, sO, h * kDh, bi * s + qb * kRows);
        tma_store_2d(&maps.o, sO + kHalf, h * kDh + 64, bi * s + qb * kRows);
        bulk_commit();
      }
    }
    if (storer) bulk_wait_all();
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
                                  float scale, float* lse, unsigned* sched, unsigned* err, cudaStream_t st) {
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
  const long long items = 1LL * b * H * (s / kRows);
  if (items == 0) return cudaSuccess;
  if (items > (1LL << 30)) return cudaErrorInvalidValue;
  const int group = heads_per_group(1LL * b * H, 4LL * s * dh);  // K and V of a head: s x dh x 2 x 2 bytes
  cudaError_t e = cudaMemsetAsync(sched, 0, sizeof(unsigned), st);  // the item counter of this launch
  if (e != cudaSuccess) return e;
  const long long grid = std::min<long long>(items, device_sm_count());  // persistent: one CTA per SM
  return launch_pdl(attn_flash_fwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kThreads), kSmem, st, maps,
                    b * H, H, s, group, scale, lse, sched, err);
}

}  // namespace lr
