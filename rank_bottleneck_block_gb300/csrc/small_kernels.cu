#include "small_kernels.cuh"

namespace lr {

// ------------------------------------------------------------------ fold
template <typename ST>
__global__ void fold_kernel(ST* out, StackSrc src, int rows_each, int rows, int cols, const ST* g) {
  pdl_wait();
  pdl_trigger();
  const int groups = cols / 8;
  const long long total = 1LL * rows * groups;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += 256LL * gridDim.x) {
    const int r = static_cast<int>(i / groups), c = static_cast<int>(i % groups) * 8;
    const ST* s = static_cast<const ST*>(src.src[r / rows_each]) + static_cast<long long>(r % rows_each) * cols;
    float v[8];
    load8(s + c, v);
    if (g) {
      float gv[8];
      load8(g + c, gv);
#pragma unroll
      for (int t = 0; t < 8; ++t) v[t] *= gv[t];
    }
    store8(out + static_cast<long long>(r) * cols + c, v);
  }
}

template <typename ST>
cudaError_t launch_fold(ST* out, StackSrc src, int nsrc, int rows_each, int cols, const ST* g, cudaStream_t st) {
  const int rows = nsrc * rows_each;
  const long long total = 1LL * rows * (cols / 8);
  if (total == 0) return cudaSuccess;
  int blocks = static_cast<int>((total + 255) / 256);
  if (blocks > 8192) blocks = 8192;
  return launch_pdl(fold_kernel<ST>, dim3(blocks), dim3(256), 0, st, out, src, rows_each, rows, cols, g);
}

// ------------------------------------------------------------------ rstd
template <typename ST>
__global__ void rstd_kernel(const ST* x, int T, int d, float eps, float* s, int raw) {
  pdl_wait();
  pdl_trigger();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  const ST* row = x + static_cast<long long>(warp) * d;
  float ss = 0.f;
  for (int j = lane * 8; j < d; j += 32 * 8) {
    float v[8];
    load8(row + j, v);
#pragma unroll
    for (int t = 0; t < 8; ++t) ss = fmaf(v[t], v[t], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) s[warp] = raw ? ss : 1.f / sqrtf(ss / static_cast<float>(d) + eps);
}

template <typename ST>
cudaError_t launch_rstd(const ST* x, int T, int d, float eps, float* s, cudaStream_t st, bool raw) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + 7) / 8;
  return launch_pdl(rstd_kernel<ST>, dim3(blocks), dim3(256), 0, st, x, T, d, eps, s, raw ? 1 : 0);
}

// ------------------------------------------------------------ norm finish
template <typename ST>
__global__ void norm_finish_kernel(const float* acc, const float* ss, int T, int n, float coef, float eps, int act,
                                   ST* u, ST* z, float* s) {
  pdl_wait();
  pdl_trigger();
  const int groups = n / 8;
  const long long total = 1LL * T * groups;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += 256LL * gridDim.x) {
    const long long t = i / groups;
    const int c = static_cast<int>(i % groups) * 8;
    const float st = rsqrtf(ss[t] * coef + eps);
    if (c == 0) s[t] = st;
    float v[8], w[8];
    load8(acc + t * n + c, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      v[q] = Num<ST>::round(st * v[q]);
      w[q] = act ? v[q] : silu<ST>(v[q]);
    }
    store8(u + t * n + c, v);
    store8(z + t * n + c, w);
  }
}

template <typename ST>
cudaError_t launch_norm_finish(const float* acc, const float* ss, int T, int n, float coef, float eps, int act, ST* u,
                               ST* z, float* s, cudaStream_t st) {
  const long long total = 1LL * T * (n / 8);
  if (total == 0) return cudaSuccess;
  int blocks = static_cast<int>((total + 255) / 256);
  if (blocks > 8192) blocks = 8192;
  return launch_pdl(norm_finish_kernel<ST>, dim3(blocks), dim3(256), 0, st, acc, ss, T, n, coef, eps, act, u, z, s);
}

// ------------------------------------------------------------------ silu
template <typename ST>
__global__ void silu_kernel(SiluSlab a, SiluSlab b, int T) {
  pdl_wait();
  pdl_trigger();
  const long long ga = 1LL * T * (a.n / 8), gb = 1LL * T * (b.n / 8);
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < ga + gb; i += 256LL * gridDim.x) {
    const bool first = i < ga;
    const SiluSlab& sl = first ? a : b;
    const long long k = first ? i : i - ga;
    const int groups = sl.n / 8;
    const long long t = k / groups;
    const int c = static_cast<int>(k % groups) * 8;
    float v[8];
    load8(static_cast<const ST*>(sl.u) + t * sl.ldu + c, v);
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = silu<ST>(v[q]);
    store8(static_cast<ST*>(sl.z) + t * sl.ldz + c, v);
  }
}

template <typename ST>
cudaError_t launch_silu(SiluSlab a, SiluSlab b, int T, cudaStream_t st) {
  const long long total = 1LL * T * (a.n / 8 + b.n / 8);
  if (total == 0) return cudaSuccess;
  int blocks = static_cast<int>((total + 255) / 256);
  if (blocks > 8192) blocks = 8192;
  return launch_pdl(silu_kernel<ST>, dim3(blocks), dim3(256), 0, st, a, b, T);
}

// ---------------------------------------------------------- wgrad reduce
// One thread per 4 consecutive columns of kReduceRows rows; splits summed in order.  The
// row loop is unrolled so the loads of all rows and splits are in flight together.
template <typename ST>
__global__ void wgrad_reduce_kernel(const float* part, int nsplit, long long split_stride, int M, int N,
                                    const ST* colscale, WgradDst dst, int rows_each, float* dgpart) {
  pdl_wait();
  pdl_trigger();
  const int n = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (n >= N) return;
  const int r0 = blockIdx.y * kReduceRows;
  float cs[4] = {1.f, 1.f, 1.f, 1.f};
  if (colscale) {
#pragma unroll
    for (int t = 0; t < 4; ++t) cs[t] = static_cast<float>(colscale[n + t]);
  }
  float4 v[kReduceRows];
#pragma unroll
  for (int i = 0; i < kReduceRows; ++i) {
    v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r0 + i < M) v[i] = *reinterpret_cast<const float4*>(part + static_cast<long long>(r0 + i) * N + n);
  }
  for (int s = 1; s < nsplit; ++s) {
#pragma unroll
    for (int i = 0; i < kReduceRows; ++i) {
      if (r0 + i < M) {
        const float4 w = *reinterpret_cast<const float4*>(part + s * split_stride + static_cast<long long>(r0 + i) * N + n);
        v[i].x += w.x;
        v[i].y += w.y;
        v[i].z += w.z;
        v[i].w += w.w;
      }
    }
  }
  float dga[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < kReduceRows; ++i) {
    const int m = r0 + i;
    if (m >= M) break;
    const int blk = m / rows_each;
    const long long local = static_cast<long long>(m - blk * rows_each) * N + n;
    *reinterpret_cast<float4*>(dst.dst[blk] + local) =
        make_float4(v[i].x * cs[0], v[i].y * cs[1], v[i].z * cs[2], v[i].w * cs[3]);
    if (dgpart) {
      const ST* aw = static_cast<const ST*>(dst.aw[blk]) + local;
      dga[0] = fmaf(v[i].x, static_cast<float>(aw[0]), dga[0]);
      dga[1] = fmaf(v[i].y, static_cast<float>(aw[1]), dga[1]);
      dga[2] = fmaf(v[i].z, static_cast<float>(aw[2]), dga[2]);
      dga[3] = fmaf(v[i].w, static_cast<float>(aw[3]), dga[3]);
    }
  }
  if (dgpart)
    *reinterpret_cast<float4*>(dgpart + static_cast<long long>(blockIdx.y) * N + n) =
        make_float4(dga[0], dga[1], dga[2], dga[3]);
}

template <typename ST>
cudaError_t launch_wgrad_reduce(const float* part, int nsplit, long long split_stride, int M, int N,
                                const ST* colscale, WgradDst dst, int rows_each, float* dgpart, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  dim3 grid((N / 4 + 127) / 128, (M + kReduceRows - 1) / kReduceRows);
  return launch_pdl(wgrad_reduce_kernel<ST>, grid, dim3(128), 0, st, part, nsplit, split_stride, M, N, colscale, dst,
                    rows_each, dgpart);
}

// 32 columns per block; the 8 thread rows each sum every 8th partial, then the 8 sums are
// added in a fixed order.
__global__ void dg_finalize_kernel(const float* dgpart, int nparts, int N, float* dg) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[8][33];
  const int n = blockIdx.x * 32 + threadIdx.x;
  float v = 0.f;
  if (n < N)
    for (int p = threadIdx.y; p < nparts; p += 8) v += dgpart[static_cast<long long>(p) * N + n];
  red[threadIdx.y][threadIdx.x] = v;
  __syncthreads();
  if (threadIdx.y == 0 && n < N) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += red[i][threadIdx.x];
    dg[n] = t;
  }
}

cudaError_t launch_dg_finalize(const float* dgpart, int nparts, int N, float* dg, cudaStream_t st) {
  if (N == 0) return cudaSuccess;
  return launch_pdl(dg_finalize_kernel, dim3((N + 31) / 32), dim3(32, 8), 0, st, dgpart, nparts, N, dg);
}

// ------------------------------------------------------------------- mse
template <typename ST>
__global__ void mse_kernel(const ST* y, const ST* t, long long n, ST* dy, float* partials) {
  pdl_wait();
  pdl_trigger();
  const float scale = 2.f / static_cast<float>(n);
  float acc = 0.f;
  const long long groups = n / 8;
  for (long long i = blockIdx.x * 256LL + threadIdx.x; i < groups; i += 256LL * gridDim.x) {
    float a[8], b[8], o[8];
    load8(y + i * 8, a);
    load8(t + i * 8, b);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float df = a[k] - b[k];
      acc = fmaf(df, df, acc);
      o[k] = scale * df;
    }
    store8(dy + i * 8, o);
  }
  __shared__ float red[256];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) partials[blockIdx.x] = red[0];
}

__global__ void mse_finalize_kernel(const float* partials, int nparts, long long n, float* loss) {
  pdl_wait();
  pdl_trigger();
  __shared__ float red[256];
  float acc = 0.f;
  for (int i = threadIdx.x; i < nparts; i += 256) acc += partials[i];
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = red[0] / static_cast<float>(n);
}

template <typename ST>
cudaError_t launch_mse(const ST* y, const ST* t, long long n, ST* dy, float* partials, int nparts, float* loss,
                       cudaStream_t st) {
  cudaError_t e = launch_pdl(mse_kernel<ST>, dim3(nparts), dim3(256), 0, st, y, t, n, dy, partials);
  if (e != cudaSuccess) return e;
  return launch_pdl(mse_finalize_kernel, dim3(1), dim3(256), 0, st, partials, nparts, n, loss);
}

// ------------------------------------------------------ wait self-test
__global__ void wait_selftest_kernel(unsigned* err, unsigned long long limit_ns) {
  pdl_wait();
  pdl_trigger();
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(a), "r"(1u) : "memory");
  const uint64_t t0 = global_timer_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(a), "r"(0u)
        : "memory");
    if (ok) return;  // never: nothing arrives on the barrier
    if (global_timer_ns() - t0 > limit_ns) {
      atomicOr(err, static_cast<unsigned>(DEV_ERR_TIMEOUT_SELFTEST));
      return;
    }
  }
}

cudaError_t launch_wait_selftest(unsigned* err, unsigned long long limit_ns, cudaStream_t st) {
  return launch_pdl(wait_selftest_kernel, dim3(1), dim3(32), 0, st, err, limit_ns);
}

// ------------------------------------------------------ instantiations
#define LR_SMALL_INST(ST)                                                                                          \
  template cudaError_t launch_fold<ST>(ST*, StackSrc, int, int, int, const ST*, cudaStream_t);                   \
  template cudaError_t launch_rstd<ST>(const ST*, int, int, float, float*, cudaStream_t, bool);                  \
  template cudaError_t launch_norm_finish<ST>(const float*, const float*, int, int, float, float, int, ST*, ST*,    \
                                              float*, cudaStream_t);                                            \
  template cudaError_t launch_silu<ST>(SiluSlab, SiluSlab, int, cudaStream_t);                                  \
  template cudaError_t launch_wgrad_reduce<ST>(const float*, int, long long, int, int, const ST*, WgradDst, int, \
                                               float*, cudaStream_t);                                            \
  template cudaError_t launch_mse<ST>(const ST*, const ST*, long long, ST*, float*, int, float*, cudaStream_t);
LR_SMALL_INST(float)
LR_SMALL_INST(bf16)
#undef LR_SMALL_INST

}  // namespace lr
