// Fused GEMM epilogues of the low-rank bottleneck sublayer.
//
// One call handles one output row m and W consecutive columns n0 .. n0+W-1 of
// one batch entry; v[a][j] is accumulator a at column n0 + j.  W is a multiple
// of 8 and every N handled here is a multiple of 8, so each 8-column group is
// either fully inside the output or fully outside it.  Row partial sums are
// accumulated over the whole W-column chunk, so each chunk writes exactly one
// partial per row (chunk index n0 / W).
//
// The math follows the unfused definition of the block (BOOST technical
// summary §2.2 states each optimisation is an exact rewrite):
//  * Online-RMSNorm: with the gain folded into A (A' = A * g), the forward
//    pre-activation is u = s * (x A'^T) with s = (mean x^2 + eps)^-1/2, and the
//    backward is dx = s (du A') - (s^2 / d) rho x with rho = sum_i du_i u_i;
//  * SwiGLU: h = SiLU(a) * b, da = dh b SiLU'(a), db = dh SiLU(a).
#pragma once

#include "common.cuh"

namespace lr {

template <EpiKind K, typename ST, int W, int NACC>
__device__ __forceinline__ void epi_apply(const EpiParams& p, int b, int split, int m, int n0,
                                          float (&v)[NACC][W]) {
  static_assert(W % 8 == 0, "chunk width must be a multiple of 8");
  if constexpr (K == EPI_NORM_SILU || K == EPI_SILU) {
    const float s = (K == EPI_NORM_SILU) ? p.rowscale[m] : 1.f;
    ST* u_out = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    ST* z_out = static_cast<ST*>(p.out1[b]) + (long long)m * p.ldo1;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float u[8], z[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          u[t] = Num<ST>::round(s * v[0][j + t]);
          z[t] = silu<ST>(u[t]);
        }
        store8(u_out + n0 + j, u);
        store8(z_out + n0 + j, z);
      }
    }
  } else if constexpr (K == EPI_STORE) {
    ST* o = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
#pragma unroll
    for (int j = 0; j < W; j += 8)
      if (n0 + j < p.N) store8(o + n0 + j, &v[0][j]);
  } else if constexpr (K == EPI_RESID) {
    ST* o = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    const ST* x = static_cast<const ST*>(p.aux0[b]) + (long long)m * p.lda0;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float xv[8], o8[8];
        load8(x + n0 + j, xv);
#pragma unroll
        for (int t = 0; t < 8; ++t) o8[t] = xv[t] + v[0][j + t];
        store8(o + n0 + j, o8);
      }
    }
  } else if constexpr (K == EPI_SWIGLU) {
    static_assert(NACC == 2, "SwiGLU needs the gate and up accumulators");
    ST* h_out = static_cast<ST*>(p.out0[0]) + (long long)m * p.ldo0;
    ST* a_out = p.out1[0] ? static_cast<ST*>(p.out1[0]) + (long long)m * p.ldo1 : nullptr;
    ST* b_out = p.out2[0] ? static_cast<ST*>(p.out2[0]) + (long long)m * p.ldo2 : nullptr;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float a[8], bb[8], h[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          a[t] = Num<ST>::round(v[0][j + t]);
          bb[t] = Num<ST>::round(v[1][j + t]);
          h[t] = silu<ST>(a[t]) * bb[t];
        }
        store8(h_out + n0 + j, h);
        if (a_out) store8(a_out + n0 + j, a);
        if (b_out) store8(b_out + n0 + j, bb);
      }
    }
  } else if constexpr (K == EPI_DSILU) {
    ST* o = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    const ST* u = static_cast<const ST*>(p.aux0[b]) + (long long)m * p.lda0;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float uv[8], du[8];
        load8(u + n0 + j, uv);
#pragma unroll
        for (int t = 0; t < 8; ++t) du[t] = v[0][j + t] * silu_grad<ST>(uv[t]);
        store8(o + n0 + j, du);
      }
    }
  } else if constexpr (K == EPI_DSILU_NORM) {
    if (n0 >= p.N) return;
    const float s = p.rowscale[m];
    ST* o = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    const ST* u = static_cast<const ST*>(p.aux0[b]) + (long long)m * p.lda0;
    float part = 0.f;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float uv[8], ds[8];
        load8(u + n0 + j, uv);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float du = v[0][j + t] * silu_grad<ST>(uv[t]);
          part = fmaf(du, uv[t], part);
          ds[t] = s * du;
        }
        store8(o + n0 + j, ds);
      }
    }
    p.rowpart[((long long)b * p.rowpart_chunks + n0 / W) * p.M + m] = part;
  } else if constexpr (K == EPI_SWIGLU_BWD) {
    ST* da_out = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    ST* db_out = static_cast<ST*>(p.out1[b]) + (long long)m * p.ldo1;
    const ST* a = static_cast<const ST*>(p.aux0[b]) + (long long)m * p.lda0;
    const ST* bb = static_cast<const ST*>(p.aux1[b]) + (long long)m * p.lda1;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float av[8], bv[8], da[8], db[8];
        load8(a + n0 + j, av);
        load8(bb + n0 + j, bv);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float dh = v[0][j + t];
          const float l = Num<ST>::logistic(av[t]);
          da[t] = dh * bv[t] * (l * (1.f + av[t] * (1.f - l)));
          db[t] = dh * (av[t] * l);
        }
        store8(da_out + n0 + j, da);
        store8(db_out + n0 + j, db);
      }
    }
  } else if constexpr (K == EPI_DX_NORM) {
    float rho = 0.f;
    for (int c = 0; c < p.rowpart_in_chunks; ++c) rho += p.rowpart_in[(long long)c * p.M + m];
    const float s = p.rowscale[m];
    const float k = p.coef * s * s * rho;
    ST* o = static_cast<ST*>(p.out0[b]) + (long long)m * p.ldo0;
    const ST* G = p.aux0[b] ? static_cast<const ST*>(p.aux0[b]) + (long long)m * p.lda0 : nullptr;
    const ST* x = static_cast<const ST*>(p.aux1[b]) + (long long)m * p.lda1;
#pragma unroll
    for (int j = 0; j < W; j += 8) {
      if (n0 + j < p.N) {
        float xv[8], gv[8], o8[8];
        load8(x + n0 + j, xv);
        if (G) {
          load8(G + n0 + j, gv);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) gv[t] = 0.f;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) o8[t] = gv[t] + v[0][j + t] - k * xv[t];
        store8(o + n0 + j, o8);
      }
    }
  } else if constexpr (K == EPI_F32) {
    float* o = static_cast<float*>(p.out0[b]) + (long long)split * p.split_stride + (long long)m * p.ldo0;
#pragma unroll
    for (int j = 0; j < W; j += 8)
      if (n0 + j < p.N) store8(o + n0 + j, &v[0][j]);
  }
}

}  // namespace lr
