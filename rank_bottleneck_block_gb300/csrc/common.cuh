// Shared device/host definitions of the low-rank bottleneck library.
//
// The sublayer is the low-rank pair of "BOOST: BOttleneck-Optimized Scalable
// Training Framework for Low-Rank Large Language Models" (technical summary §1
// and §2.1: each dense map becomes an r x d_in layer followed by a d_out x r
// layer), read as y = B . SiLU(A . v).  Every GEMM of the forward and backward
// pass is C[M,N] = sum_k A[m,k] B[n,k] with fp32 accumulation, followed by one
// of the fused epilogues enumerated in EpiKind.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <utility>

namespace lr {

using bf16 = __nv_bfloat16;

// Epilogues fused into the GEMMs.  "acc" is the fp32 accumulator of the tile,
// "round" rounds to the storage type before the value is used again, so a
// re-forward from saved tensors reproduces the forward bit for bit.
enum EpiKind : int {
  EPI_NORM_SILU = 0,  // u = round(s[m] * acc) -> out0, z = SiLU(u) -> out1          (online RMSNorm)
  EPI_SILU = 1,       // u = round(acc) -> out0,  z = SiLU(u) -> out1                (plain A GEMM)
  EPI_STORE = 2,      // out0 = acc                                                  (B GEMM)
  EPI_RESID = 3,      // out0 = aux0 + acc                                           (B_down + residual)
  EPI_SWIGLU = 4,     // two accumulators: a, b; h = SiLU(a) * b -> out0, a -> out1, b -> out2 (optional)
  EPI_DSILU = 5,      // out0 = acc * SiLU'(aux0)                                    (du of a plain pair)
  EPI_DSILU_NORM = 6, // du = acc * SiLU'(aux0); out0 = s[m] * du; rowpart = sum du * aux0
  EPI_SWIGLU_BWD = 7, // dh = acc; a = aux0, b = aux1: out0 = dh b SiLU'(a), out1 = dh SiLU(a)
  EPI_DX_NORM = 8,    // out0 = aux0 (optional) + acc - coef s[m]^2 rho[m] aux1[m,n], rho = sum of rowpart_in
  EPI_F32 = 9,        // fp32 out0 (+ split * split_stride): weight-gradient partials
  EPI_NORM_SWIGLU = 10,     // dense gate/up: a = round(s acc0), b = round(s acc1), h = SiLU(a) b -> (h, a, b)
  EPI_SWIGLU_BWD_NORM = 11, // dense: dh = acc; da, db as SWIGLU_BWD; out0 = s da, out1 = s db;
                            //        rowpart = sum (da a + db b)
  EPI_F32_SS = 12,          // fp32 out0 = acc (no split); the row sums of squares of the A tiles (raw,
                            //   not 1/rms) -> rowscale_out: the partial of a row-parallel normed GEMM
  EPI_ATTN_BWD = 13,        // causal attention backward scores, row-batched over heads: acc0 = Q K^T,
                            //   acc1 = dO V^T; out0 = P = exp(coef acc0 - lse) (0 past the diagonal),
                            //   out1 = dS = coef P (acc1 - D); lse = rowscale, D = rowpart_in (global rows)
  EPI_SWIGLU_REBWD = 14,    // checkpointed re-forward and SwiGLU backward of one tile: three accumulators
                            //   a = round(acc0), b = round(acc1), dh = acc2; h = SiLU(a) b -> out0,
                            //   da = dh b SiLU'(a) -> out1, db = dh SiLU(a) -> out2
  EPI_SWIGLU_H = 15,        // EPI_SWIGLU storing h only (the forward of the checkpointed block)
  EPI_DSILU_Z = 16,         // EPI_DSILU that also writes z = SiLU(aux0) -> out1 (the checkpointed backward's
                            //   re-forward of z_down from the saved u_down, which the epilogue reads anyway)
  EPI_COUNT = 17
};

constexpr int kMaxBatch = 4;

// Everything an epilogue may read or write.  Pointers indexed by the batch
// entry (or by the accumulator for the dual-accumulator epilogue).
struct EpiParams {
  int M, N;                       // extent of one batch entry's output
  void* out0[kMaxBatch];
  void* out1[kMaxBatch];
  void* out2[kMaxBatch];
  long long ldo0, ldo1, ldo2;     // leading dimensions (elements)
  const void* aux0[kMaxBatch];
  const void* aux1[kMaxBatch];
  long long lda0, lda1;
  const float* rowscale;          // s[m] = 1/rms of row m
  float* rowpart;                 // [batches * chunks_per_batch][M] row partial sums (written)
  int rowpart_chunks;             // chunks per batch entry = ceil(N / chunk width)
  const float* rowpart_in;        // [rowpart_in_chunks][M] (read, summed in order)
  int rowpart_in_chunks;
  float coef;                     // 1/d (RMSNorm forward statistics and backward)
  float eps;                      // RMSNorm epsilon (forward statistics)
  float* rowscale_out;            // s[m] written by the GEMM that computes it (online RMSNorm), or null
  long long split_stride;         // elements between split-K partial outputs
  int act;                        // pair activation sigma: 0 SiLU, 1 identity
};

// ---------------------------------------------------------------- numerics
template <typename ST>
struct Num;

template <>
struct Num<bf16> {
  static __device__ __forceinline__ float round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }
  // logistic(u) = 1 / (1 + e^-u) = (1 + tanh(u / 2)) / 2, with the hardware tanh approximation (one
  // special-function op instead of an exponential and a reciprocal; its error, below 2^-10 absolute on
  // the logistic, is far under bf16 storage precision).  tanh saturates to -1 / +1 for large |u|, so
  // the logistic reaches exactly 0 / 1 there.
  static __device__ __forceinline__ float logistic(float u) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * u));
    return fmaf(0.5f, t, 0.5f);
  }
};

template <>
struct Num<float> {
  static __device__ __forceinline__ float round(float v) { return v; }
  static __device__ __forceinline__ float logistic(float u) { return 1.f / (1.f + expf(-u)); }
};

template <typename ST>
__device__ __forceinline__ float silu(float u) { return u * Num<ST>::logistic(u); }

template <typename ST>
__device__ __forceinline__ float silu_grad(float u) {
  const float l = Num<ST>::logistic(u);
  return l * (1.f + u * (1.f - l));
}

// 8-wide vector loads / stores (16 bytes of bf16, 32 bytes of fp32).
__device__ __forceinline__ void load8(const bf16* p, float* v) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
    const float2 f = __bfloat1622float2(h);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* v) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void store8(bf16* p, const float* v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float* p, const float* v) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ------------------------------------------------------------ error word
// Bits of the device error word that kernels set instead of trapping.
enum DeviceError : unsigned {
  DEV_ERR_TIMEOUT_PRODUCER = 1u,
  DEV_ERR_TIMEOUT_MMA = 2u,
  DEV_ERR_TIMEOUT_EPILOGUE = 4u,
  DEV_ERR_TIMEOUT_SELFTEST = 8u,
  DEV_ERR_TMEM = 16u,
};

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------- programmatic dependent launch
// Every kernel of the library is launched with programmatic stream
// serialisation: it may start (and run its prologue) while the kernel before it
// in the stream is still finishing.  pdl_wait() returns once that kernel has
// completed and its memory operations are visible; every thread calls it before
// its first global-memory access and before any early return (so a grid never
// completes ahead of its predecessor and the ordering stays transitive).
// pdl_trigger() lets the next kernel be scheduled once every CTA of this grid has
// called it or exited; it does not release any memory ordering.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launches issued on this host thread while a PdlOff guard lives carry no programmatic-launch
// attribute (each kernel then starts after the previous one has completed).
inline int& pdl_suppressed() {
  static thread_local int n = 0;
  return n;
}
struct PdlOff {
  PdlOff() { ++pdl_suppressed(); }
  ~PdlOff() { --pdl_suppressed(); }
  PdlOff(const PdlOff&) = delete;
  PdlOff& operator=(const PdlOff&) = delete;
};

// Programmatic dependent launch is on unless the environment sets LR_PDL=0 (read once) or a
// PdlOff guard is active.
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = getenv("LR_PDL");
    return !(e && e[0] == '0');
  }();
  return on && pdl_suppressed() == 0;
}

// Launches kern<<<grid, block, smem, st>>>(args...) with the programmatic-serialisation attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace lr
