// Small memory-bound kernels around the GEMMs: gain folding / stacking of A,
// the per-row inverse rms, SiLU of saved pre-activations, the deterministic
// split-K reduction of weight gradients (with the gain unfold and the dg
// column reduction), the MSE loss, and a self-test of the bounded wait.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace lr {

constexpr int kMaxStack = 3;

struct StackSrc {
  const void* src[kMaxStack];  // each [rows_each, cols]
};

struct WgradDst {
  float* dst[kMaxStack];         // each [rows_each, N] fp32
  const void* aw[kMaxStack];     // unfolded A row blocks for dg (storage dtype), or null
};

// out[i, j] = src[i / rows_each][i % rows_each, j] * (g ? g[j] : 1), rounded to the storage type.
template <typename ST>
cudaError_t launch_fold(ST* out, StackSrc src, int nsrc, int rows_each, int cols, const ST* g, cudaStream_t st);

// s[t] = (sum_j x[t, j]^2 / d + eps)^(-1/2), or with `raw` the sum of squares itself; one warp per row.
template <typename ST>
cudaError_t launch_rstd(const ST* x, int T, int d, float eps, float* s, cudaStream_t st, bool raw = false);

// Finish of a row-parallel normed group from its all-reduced fp32 partials acc [T, n] and row sums of
// squares ss [T]: s = (ss coef + eps)^(-1/2), u = round(s acc), z = sigma(u) (act 0 SiLU, 1 identity).
template <typename ST>
cudaError_t launch_norm_finish(const float* acc, const float* ss, int T, int n, float coef, float eps, int act, ST* u,
                               ST* z, float* s, cudaStream_t st);

// z[t, j] = SiLU(u[t, j]) for two [T, n] slabs in one launch (u and z with their own leading
// dimensions; a slab with n = 0 is skipped).
struct SiluSlab {
  const void* u;
  long long ldu;
  void* z;
  long long ldz;
  int n;
};
template <typename ST>
cudaError_t launch_silu(SiluSlab a, SiluSlab b, int T, cudaStream_t st);

// dst = sum over splits of part (fixed order) times the optional column scale;
// dgpart[row_block, n] = sum over the block's rows of (unscaled sum) * aw.
template <typename ST>
cudaError_t launch_wgrad_reduce(const float* part, int nsplit, long long split_stride, int M, int N,
                                const ST* colscale, WgradDst dst, int rows_each, float* dgpart, cudaStream_t st);
constexpr int kReduceRows = 8;

// dg[n] = sum_p dgpart[p, n].
cudaError_t launch_dg_finalize(const float* dgpart, int nparts, int N, float* dg, cudaStream_t st);

// loss = mean((y - t)^2) (fp32, deterministic), dy = 2 (y - t) / n.
template <typename ST>
cudaError_t launch_mse(const ST* y, const ST* t, long long n, ST* dy, float* partials, int nparts, float* loss,
                       cudaStream_t st);
constexpr int kMseParts = 1024;

// Bounded-wait self-test: waits on an mbarrier that nothing completes for
// `limit_ns`, then sets DEV_ERR_TIMEOUT_SELFTEST in *err and returns.
cudaError_t launch_wait_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t st);

}  // namespace lr
