"""fp64 CPU oracle for causal multi-head self-attention between the low-rank projections.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may call
it.  It shares no code with the CUDA library.

The BOOST technical summary trains low-rank LLaMA-style transformers: the attention
projections q, k, v and o are the low-rank pairs of the projection groups, and between
them sits ordinary causal softmax attention, which the method leaves unchanged.  This file
is that attention written out by its textbook definition, per batch entry and head:

    S = scale * Q K^T,  S_ij = -inf for j > i (causal),  P = softmax_j(S),  O = P V,

with the log-sum-exp of every row, lse_i = log sum_j exp(S_ij), kept for the backward.
Gradients by the chain rule through the softmax:

    dV = P^T dO,  dP = dO V^T,  D_i = sum_j P_ij dP_ij,  dS = P * (dP - D),
    dQ = scale * dS K,  dK = scale * dS^T Q.

Tensors are token-major as the projections produce them: q, k, v, o are [b*s, H*dh] with
head h of token t in columns h*dh .. h*dh + dh - 1 of row t.  float64 throughout; matrix
products use numpy's ``@`` (a library primitive).

The full low-rank transformer block composes this attention with the projection groups and
the MLP block of ``lowrank_oracle`` (pre-norm residual form, as in LLaMA):

    [q; k; v] = LR_{q,k,v}(RMSNorm_a(x)),  y = LR_o(attention(q, k, v)),  x1 = x + y,
    out = x1 + LR_down(SiLU(LR_gate(n1)) * LR_up(n1)),  n1 = RMSNorm_m(x1),

and its backward chains the pieces' backward functions, the residual adding its gradient.

Pins (tests/test_attention_oracle.py): a brute-force triple loop on tiny sizes, central finite
differences of every gradient (of the attention and of the whole block), causality (later keys
and values do not change earlier outputs), the first token's output equals its own value, and
q = 0 gives the running mean of the values.  No function here is parity unpinned.
"""
from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

F64 = np.float64

__all__ = ["heads", "unheads", "attention_fwd", "attention_bwd", "block_fwd", "block_bwd"]


def heads(x: np.ndarray, b: int, s: int, H: int, dh: int) -> np.ndarray:
    """[b*s, H*dh] token-major -> [b, H, s, dh]."""
    return np.asarray(x, dtype=F64).reshape(b, s, H, dh).transpose(0, 2, 1, 3)


def unheads(x: np.ndarray) -> np.ndarray:
    """[b, H, s, dh] -> [b*s, H*dh]."""
    b, H, s, dh = x.shape
    return x.transpose(0, 2, 1, 3).reshape(b * s, H * dh)


def _causal_mask(s: int) -> np.ndarray:
    return np.triu(np.ones((s, s), dtype=bool), k=1)  # True where key j > query i


def attention_fwd(q, k, v, b: int, s: int, H: int, dh: int, scale: float) -> Tuple[np.ndarray, Dict]:
    """Causal softmax attention.  Returns o [b*s, H*dh] and the saved row log-sum-exp
    lse [b, H, s]."""
    Q, K, V = heads(q, b, s, H, dh), heads(k, b, s, H, dh), heads(v, b, s, H, dh)
    S = scale * (Q @ K.transpose(0, 1, 3, 2))
    S = np.where(_causal_mask(s), -np.inf, S)
    m = S.max(axis=-1, keepdims=True)
    E = np.exp(S - m)
    l = E.sum(axis=-1, keepdims=True)
    P = E / l
    O = P @ V
    lse = (m + np.log(l))[..., 0]
    return unheads(O), {"lse": lse}


def attention_bwd(q, k, v, o, saved: Dict, do, b: int, s: int, H: int, dh: int, scale: float):
    """Gradients of sum(o * do) with respect to q, k, v (each [b*s, H*dh])."""
    Q, K, V = heads(q, b, s, H, dh), heads(k, b, s, H, dh), heads(v, b, s, H, dh)
    O, dO = heads(o, b, s, H, dh), heads(do, b, s, H, dh)
    S = scale * (Q @ K.transpose(0, 1, 3, 2))
    S = np.where(_causal_mask(s), -np.inf, S)
    P = np.exp(S - saved["lse"][..., None])
    dV = P.transpose(0, 1, 3, 2) @ dO
    dP = dO @ V.transpose(0, 1, 3, 2)
    D = np.sum(dO * O, axis=-1, keepdims=True)
    dS = P * (dP - D)
    dQ = scale * (dS @ K)
    dK = scale * (dS.transpose(0, 1, 3, 2) @ Q)
    return {"dq": unheads(dQ), "dk": unheads(dK), "dv": unheads(dV)}


# ---------------------------------------------------------------------------
# The full low-rank transformer block.
# ---------------------------------------------------------------------------
def block_fwd(x, W: Dict, b: int, s: int, H: int, dh: int, scale: float, eps: float = 1e-6):
    """W: g_attn, A_q/B_q, A_k/B_k, A_v/B_v, A_o/B_o, g_mlp and the MLP's A_*/B_* (gate, up,
    down).  Returns (out, saved)."""
    from . import lowrank_oracle as O

    x = O.to64(x)
    qkv, s_qkv = O.proj_group_fwd(x, W["g_attn"], [W["A_q"], W["A_k"], W["A_v"]],
                                  [W["B_q"], W["B_k"], W["B_v"]], eps)
    o, s_att = attention_fwd(qkv[0], qkv[1], qkv[2], b, s, H, dh, scale)
    (y,), s_o = O.proj_group_fwd(o, None, [W["A_o"]], [W["B_o"]], eps)
    x1 = x + y
    mlp = {k: W[k] for k in ("A_gate", "B_gate", "A_up", "B_up", "A_down", "B_down")}
    out, s_mlp = O.mlp_block_fwd(x1, W["g_mlp"], mlp, eps, O.FULL)
    return out, dict(qkv=qkv, s_qkv=s_qkv, o=o, s_att=s_att, s_o=s_o, mlp=mlp, s_mlp=s_mlp)


def block_bwd(W: Dict, saved: Dict, G, b: int, s: int, H: int, dh: int, scale: float, eps: float = 1e-6):
    """Gradients of sum(out * G): dx, dg_attn, dg_mlp, and dA_*/dB_* for q, k, v, o, gate,
    up, down."""
    from . import lowrank_oracle as O

    gm = O.mlp_block_bwd(W["g_mlp"], saved["mlp"], saved["s_mlp"], O.to64(G), eps)
    dx1 = gm["dx"]  # includes the residual path of the MLP block
    go = O.proj_group_bwd(None, [W["A_o"]], [W["B_o"]], saved["s_o"], [dx1])
    q, k, v = saved["qkv"]
    ga = attention_bwd(q, k, v, saved["o"], saved["s_att"], go["dx"], b, s, H, dh, scale)
    gq = O.proj_group_bwd(W["g_attn"], [W["A_q"], W["A_k"], W["A_v"]], [W["B_q"], W["B_k"], W["B_v"]],
                          saved["s_qkv"], [ga["dq"], ga["dk"], ga["dv"]])
    out = {"dx": dx1 + gq["dx"], "dg_attn": gq["dg"], "dg_mlp": gm["dg"]}
    for i, n in enumerate("qkv"):
        out[f"dA_{n}"], out[f"dB_{n}"] = gq["dA"][i], gq["dB"][i]
    out["dA_o"], out["dB_o"] = go["dA"][0], go["dB"][0]
    for n in ("gate", "up", "down"):
        out[f"dA_{n}"], out[f"dB_{n}"] = gm[f"dA_{n}"], gm[f"dB_{n}"]
    return out
