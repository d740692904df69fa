// Fused GEMM epilogues of the low-rank bottleneck sublayer.
//
// EpiDef<K> describes one epilogue: how many accumulators it consumes (NACC),
// how many same-shaped operand tiles it reads besides them (NAUX), how many
// output tiles it writes (NOUT, bf16/fp32 per the storage type, or fp32 for the
// weight-gradient partials), which per-row scalars it needs, and its math on W
// consecutive columns of one row.  Both GEMM engines share this math; only the
// way operand and output tiles move differs (TMA tiles through shared memory in
// the tcgen05 kernel, direct global accesses in the SIMT kernel).
//
// The math follows the unfused definition of the block (BOOST technical
// summary §2.2 states each optimisation is an exact rewrite):
//  * Online-RMSNorm: with the gain folded into A (A' = A * g), the forward
//    pre-activation is u = s * (x A'^T) with s = (mean x^2 + eps)^-1/2, and the
//    backward is dx = s (du A') - (s^2 / d) rho x with rho = sum_i du_i u_i;
//  * SwiGLU: h = SiLU(a) * b, da = dh b SiLU'(a), db = dh SiLU(a).
// Values that are stored and used again are rounded to the storage type first,
// so a re-forward from saved tensors reproduces the forward bit for bit.
#pragma once

#include "common.cuh"

namespace lr {

// Per-row inputs of an epilogue: s = 1/rms of the row, k = coef * s^2 * rho, and the pair
// activation (0 SiLU, 1 identity; uniform over the launch).
struct RowIn {
  float s;
  float k;
  int act;
};

// The pair activation sigma and its derivative.
template <typename ST>
__device__ __forceinline__ float pair_act(int act, float u) {
  return act ? u : silu<ST>(u);
}
template <typename ST>
__device__ __forceinline__ float pair_act_grad(int act, float u) {
  return act ? 1.f : silu_grad<ST>(u);
}

template <EpiKind K>
struct EpiDef;

template <>
struct EpiDef<EPI_NORM_SILU> {  // u = round(s acc), z = sigma(u)
  static constexpr int NACC = 1, NAUX = 0, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = true, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&)[1][W],
                                             float (&o)[2][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float u = Num<ST>::round(ri.s * v[0][j]);
      o[0][j] = u;
      o[1][j] = pair_act<ST>(ri.act, u);
    }
  }
};

template <>
struct EpiDef<EPI_SILU> {  // u = round(acc), z = sigma(u)
  static constexpr int NACC = 1, NAUX = 0, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&)[1][W],
                                             float (&o)[2][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float u = Num<ST>::round(v[0][j]);
      o[0][j] = u;
      o[1][j] = pair_act<ST>(ri.act, u);
    }
  }
};

template <>
struct EpiDef<EPI_STORE> {  // out = acc
  static constexpr int NACC = 1, NAUX = 0, NOUT = 1;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[1][W], const float (&)[1][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = v[0][j];
  }
};

template <>
struct EpiDef<EPI_RESID> {  // out = x + acc  (aux0 = x)
  static constexpr int NACC = 1, NAUX = 1, NOUT = 1;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[1][W], const float (&a)[1][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = a[0][j] + v[0][j];
  }
};

template <>
struct EpiDef<EPI_SWIGLU> {  // a = round(acc0), b = round(acc1), h = SiLU(a) b -> (h, a, b)
  static constexpr int NACC = 2, NAUX = 0, NOUT = 3;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[2][W], const float (&)[1][W],
                                             float (&o)[3][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float a = Num<ST>::round(v[0][j]);
      const float b = Num<ST>::round(v[1][j]);
      o[0][j] = silu<ST>(a) * b;
      o[1][j] = a;
      o[2][j] = b;
    }
  }
};

template <>
struct EpiDef<EPI_SWIGLU_H> : EpiDef<EPI_SWIGLU> {  // h = SiLU(round(acc0)) round(acc1) only
  static constexpr int NOUT = 1;
};

template <>
struct EpiDef<EPI_DSILU> {  // du = acc sigma'(u)  (aux0 = u)
  static constexpr int NACC = 1, NAUX = 1, NOUT = 1;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&a)[1][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = v[0][j] * pair_act_grad<ST>(ri.act, a[0][j]);
  }
};

template <>
struct EpiDef<EPI_DSILU_Z> {  // du = acc sigma'(u), z = sigma(u)  (aux0 = u)
  static constexpr int NACC = 1, NAUX = 1, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&a)[1][W],
                                             float (&o)[2][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      o[0][j] = v[0][j] * pair_act_grad<ST>(ri.act, a[0][j]);
      o[1][j] = pair_act<ST>(ri.act, a[0][j]);
    }
  }
};

template <>
struct EpiDef<EPI_DSILU_NORM> {  // du = acc sigma'(u); out = s du; row partial += du u  (aux0 = u)
  static constexpr int NACC = 1, NAUX = 1, NOUT = 1;
  static constexpr bool OUT_F32 = false, NEED_S = true, NEED_RHO = false, ROWPART = true;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&a)[1][W],
                                             float (&o)[1][W], float& part) {
    float p = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float du = v[0][j] * pair_act_grad<ST>(ri.act, a[0][j]);
      p = fmaf(du, a[0][j], p);
      o[0][j] = ri.s * du;
    }
    part = p;
  }
};

template <>
struct EpiDef<EPI_SWIGLU_BWD> {  // dh = acc; da = dh b SiLU'(a), db = dh SiLU(a)  (aux0 = a, aux1 = b)
  static constexpr int NACC = 1, NAUX = 2, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[1][W], const float (&a)[2][W],
                                             float (&o)[2][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float dh = v[0][j], av = a[0][j], bv = a[1][j];
      const float l = Num<ST>::logistic(av);
      o[0][j] = dh * bv * (l * (1.f + av * (1.f - l)));
      o[1][j] = dh * (av * l);
    }
  }
};

template <>
struct EpiDef<EPI_DX_NORM> {  // dx = G + acc - k x  (aux0 = G, may be absent; aux1 = x)
  static constexpr int NACC = 1, NAUX = 2, NOUT = 1;
  static constexpr bool OUT_F32 = false, NEED_S = true, NEED_RHO = true, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&a)[2][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = a[0][j] + v[0][j] - ri.k * a[1][j];
  }
};

template <>
struct EpiDef<EPI_NORM_SWIGLU> {  // a = round(s acc0), b = round(s acc1), h = SiLU(a) b -> (h, a, b)
  static constexpr int NACC = 2, NAUX = 0, NOUT = 3;
  static constexpr bool OUT_F32 = false, NEED_S = true, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[2][W], const float (&)[1][W],
                                             float (&o)[3][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float a = Num<ST>::round(ri.s * v[0][j]);
      const float b = Num<ST>::round(ri.s * v[1][j]);
      o[0][j] = silu<ST>(a) * b;
      o[1][j] = a;
      o[2][j] = b;
    }
  }
};

template <>
struct EpiDef<EPI_SWIGLU_BWD_NORM> {  // dh = acc; da, db; out = s da, s db; part = sum da a + db b (aux a, b)
  static constexpr int NACC = 1, NAUX = 2, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = true, NEED_RHO = false, ROWPART = true;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn& ri, const float (&v)[1][W], const float (&a)[2][W],
                                             float (&o)[2][W], float& part) {
    float p = 0.f;
#pragma unroll
    for (int j = 0; j < W; ++j) {
      const float dh = v[0][j], av = a[0][j], bv = a[1][j];
      const float l = Num<ST>::logistic(av);
      const float da = dh * bv * (l * (1.f + av * (1.f - l)));
      const float db = dh * (av * l);
      p = fmaf(da, av, fmaf(db, bv, p));
      o[0][j] = ri.s * da;
      o[1][j] = ri.s * db;
    }
    part = p;
  }
};

template <>
struct EpiDef<EPI_F32_SS> {  // fp32 partial sums of a row-parallel GEMM (its row statistics come from the ring)
  static constexpr int NACC = 1, NAUX = 0, NOUT = 1;
  static constexpr bool OUT_F32 = true, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[1][W], const float (&)[1][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = v[0][j];
  }
};

template <>
struct EpiDef<EPI_ATTN_BWD> {  // P and dS of causal attention (the math lives in the split-phase epilogue)
  static constexpr int NACC = 2, NAUX = 0, NOUT = 2;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
};

template <>
struct EpiDef<EPI_SWIGLU_REBWD> {  // h, da, db of a tile from a, b, dh (the math lives in the split-phase epilogue)
  static constexpr int NACC = 3, NAUX = 0, NOUT = 3;
  static constexpr bool OUT_F32 = false, NEED_S = false, NEED_RHO = false, ROWPART = false;
};

template <>
struct EpiDef<EPI_F32> {  // fp32 weight-gradient partial
  static constexpr int NACC = 1, NAUX = 0, NOUT = 1;
  static constexpr bool OUT_F32 = true, NEED_S = false, NEED_RHO = false, ROWPART = false;
  template <typename ST, int W>
  static __device__ __forceinline__ void run(const RowIn&, const float (&v)[1][W], const float (&)[1][W],
                                             float (&o)[1][W], float&) {
#pragma unroll
    for (int j = 0; j < W; ++j) o[0][j] = v[0][j];
  }
};

// Per-row inputs of the epilogue for row m (0 for rows past the end).
template <EpiKind K>
__device__ __forceinline__ RowIn row_inputs(const EpiParams& p, int m) {
  using D = EpiDef<K>;
  RowIn ri{0.f, 0.f, p.act};
  if (m >= p.M) return ri;
  if constexpr (D::NEED_S) ri.s = p.rowscale[m];
  if constexpr (D::NEED_RHO) {
    float rho = 0.f;
    for (int c = 0; c < p.rowpart_in_chunks; ++c) rho += p.rowpart_in[(long long)c * p.M + m];
    ri.k = p.coef * ri.s * ri.s * rho;
  }
  return ri;
}

__device__ __forceinline__ const void* epi_aux_ptr(const EpiParams& p, int a, int b) {
  return a == 0 ? p.aux0[b] : p.aux1[b];
}
__device__ __forceinline__ void* epi_out_ptr(const EpiParams& p, int o, int b) {
  return o == 0 ? p.out0[b] : (o == 1 ? p.out1[b] : p.out2[b]);
}
__device__ __forceinline__ long long epi_aux_ld(const EpiParams& p, int a) { return a == 0 ? p.lda0 : p.lda1; }
__device__ __forceinline__ long long epi_out_ld(const EpiParams& p, int o) {
  return o == 0 ? p.ldo0 : (o == 1 ? p.ldo1 : p.ldo2);
}

}  // namespace lr
