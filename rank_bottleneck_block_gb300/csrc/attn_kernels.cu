// Row kernels of causal multi-head attention (see attn_kernels.cuh).
#include "attn_kernels.cuh"

namespace lr {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
// Rows of the pair tiles of the attention GEMMs: P and dS are written up to the end of the row's
// tile of keys (the GEMMs that read them stop their K range there or start it at the tile).
constexpr int kTileRows = 256;
constexpr float kLn2 = 0.6931471805599453f;

// Combines two (max, sum) pairs of a streaming log-sum-exp in base 2; an empty pair is (-inf, 0).
__device__ __forceinline__ void lse_merge(float& m, float& l, float m2, float l2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  l = (m == -INFINITY ? 0.f : l * exp2f(m - M)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - M));
  m = M;
}

__device__ __forceinline__ void store_bf16x4(bf16* p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&lo);
  u.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(p) = u;
}

// Rows of any length: one warp per row; lanes take 4 consecutive columns at a time, a streaming
// log-sum-exp first, then P from a second read of the row.
__global__ void attn_softmax_fwd_kernel(const float* S, int R, int s, float scale, bf16* P, float* lse) {
  pdl_wait();
  pdl_trigger();
  const int r = static_cast<int>((blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  const int n = r % s + 1;  // keys visible to this query
  const float* row = S + 1LL * r * s;
  const float c = scale * kLog2e;
  float m = -INFINITY, l = 0.f;
  for (int j = lane * 4; j < n; j += 128) {
    const float4 v = *reinterpret_cast<const float4*>(row + j);
    const float x[4] = {v.x * c, v.y * c, v.z * c, v.w * c};
#pragma unroll
    for (int t = 0; t < 4; ++t)
      if (j + t < n) lse_merge(m, l, x[t], 1.f);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
    lse_merge(m, l, m2, l2);
  }
  const float lse2 = m + log2f(l);
  if (lane == 0) lse[r] = lse2 * kLn2;
  bf16* prow = P + 1LL * r * s;
  const int wend = min(s, ((n - 1) / kTileRows + 1) * kTileRows);  // zeros past n up to the tile end
  for (int j = lane * 4; j < wend; j += 128) {
    float p[4] = {0.f, 0.f, 0.f, 0.f};
    if (j < n) {
      const float4 v = *reinterpret_cast<const float4*>(row + j);
      const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int t = 0; t < 4; ++t)
        if (j + t < n) p[t] = exp2f(x[t] * c - lse2);
    }
    store_bf16x4(prow + j, p[0], p[1], p[2], p[3]);
  }
}

// Rows of up to kRegKeys keys: each lane keeps its columns of S in registers, so S is read once
// and every element takes one exp2: P = 2^(c S - m) / l with m the row maximum of c S and l the
// row sum of 2^(c S - m).
constexpr int kRegVec = 16;              // float4 per lane
constexpr int kRegKeys = kRegVec * 128;  // 2048
__global__ void __launch_bounds__(128, 4) attn_softmax_fwd_reg_kernel(const float* S, int R, int s, float scale, bf16* P, float* lse) {
  pdl_wait();
  pdl_trigger();
  const int r = static_cast<int>((blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= R) return;
  const int n = r % s + 1;
  const float* row = S + 1LL * r * s;
  const float c = scale * kLog2e;
  float x[kRegVec][4];  // c S, -inf past the diagonal (so 2^(x - m) is 0 there)
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) {
    const int j = (k * 32 + lane) * 4;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < n) v = *reinterpret_cast<const float4*>(row + j);
    x[k][0] = j < n ? v.x * c : -INFINITY;
    x[k][1] = j + 1 < n ? v.y * c : -INFINITY;
    x[k][2] = j + 2 < n ? v.z * c : -INFINITY;
    x[k][3] = j + 3 < n ? v.w * c : -INFINITY;
  }
  float m = -INFINITY;
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) m = fmaxf(fmaxf(m, fmaxf(x[k][0], x[k][1])), fmaxf(x[k][2], x[k][3]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) {
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      x[k][t] = exp2f(x[k][t] - m);
      l += x[k][t];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  if (lane == 0) lse[r] = (m + log2f(l)) * kLn2;
  const float inv = 1.f / l;
  bf16* prow = P + 1LL * r * s;
  const int wend = min(s, ((n - 1) / kTileRows + 1) * kTileRows);  // zeros past n up to the tile end
#pragma unroll
  for (int k = 0; k < kRegVec; ++k) {
    const int j = (k * 32 + lane) * 4;
    if (j < wend) store_bf16x4(prow + j, x[k][0] * inv, x[k][1] * inv, x[k][2] * inv, x[k][3] * inv);
  }
}

// G lanes per row (32 when dh is a multiple of 256, else 16: dh is a multiple of 128), 32 / G rows
// per warp; each lane takes 8 consecutive channels at a time.
template <int G>
__global__ void attn_rowdot_kernel(const bf16* dO, const bf16* O, int b, int s, int H, int dh, float* D) {
  pdl_wait();
  pdl_trigger();
  const int R = b * H * s;
  const long long gt = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
  const int r = static_cast<int>(gt / G);
  const int sub = threadIdx.x & (G - 1);
  if (r >= R) return;  // whole lane groups leave together (R rows of G lanes each)
  const int n = r / s, i = r - n * s;  // head n = bi*H + h, query i
  const int bi = n / H, h = n - bi * H;
  const long long base = (1LL * bi * s + i) * H * dh + 1LL * h * dh;
  float acc = 0.f;
  for (int c = sub * 8; c < dh; c += G * 8) {
    float a[8], o[8];
    load8(dO + base + c, a);
    load8(O + base + c, o);
#pragma unroll
    for (int t = 0; t < 8; ++t) acc = fmaf(a[t], o[t], acc);
  }
  const unsigned mask = G == 32 ? 0xffffffffu : (((1u << G) - 1u) << (threadIdx.x & 31 & ~(G - 1)));
#pragma unroll
  for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(mask, acc, off);
  if (sub == 0) D[r] = acc;
}

dim3 warp_rows_grid(int R) { return dim3(static_cast<unsigned>((R + 7) / 8)); }

}  // namespace

cudaError_t launch_attn_softmax_fwd(const float* S, int R, int s, float scale, bf16* P, float* lse,
                                    cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  if (s <= kRegKeys)
    return launch_pdl(attn_softmax_fwd_reg_kernel, dim3(static_cast<unsigned>((R + 3) / 4)), dim3(128), 0, st, S, R,
                      s, scale, P, lse);
  return launch_pdl(attn_softmax_fwd_kernel, warp_rows_grid(R), dim3(256), 0, st, S, R, s, scale, P, lse);
}

cudaError_t launch_attn_rowdot(const bf16* dO, const bf16* O, int b, int s, int H, int dh, float* D,
                               cudaStream_t st) {
  const int R = b * H * s;
  if (R == 0) return cudaSuccess;
  if (dh % 256 == 0)  // a warp per row
    return launch_pdl(attn_rowdot_kernel<32>, warp_rows_grid(R), dim3(256), 0, st, dO, O, b, s, H, dh, D);
  // dh = 128 (mod 256): a half warp per row, 16 rows per block of 256 threads
  return launch_pdl(attn_rowdot_kernel<16>, dim3(static_cast<unsigned>((R + 15) / 16)), dim3(256), 0, st, dO, O, b,
                    s, H, dh, D);
}

}  // namespace lr
