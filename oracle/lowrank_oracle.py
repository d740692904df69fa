"""fp64 CPU oracle for the low-rank bottleneck sublayer (BOOST).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

What it computes is the plain, unfused definition of the sublayer described in
"BOOST: BOttleneck-Optimized Scalable Training Framework for Low-Rank Large
Language Models" (gist.science technical summary, and the arXiv abstract):

* every dense map W.x of the model is replaced by a low-rank bottleneck pair,
  an r x d_in layer A followed by a d_out x r layer B (technical summary §1 and
  §2.1: "a pair of d x r and r x d layers"); this library's reading of the pair
  is y = B . sigma(A . v) with sigma = SiLU;
* the MLP block is out = x + LR_down(SiLU(LR_gate(n)) * LR_up(n)) with
  n = RMSNorm(x) and LR(v) = B . SiLU(A . v);
* an attention-projection group is q_i = LR_i(RMSNorm(x)), and the o-projection
  is a single pair applied without a norm;
* a stack is L residual MLP blocks followed by a mean-squared error.

The three system optimisations of technical summary §2.2 are exact rewrites of
this definition: Online-RMSNorm (folding the gain into A and applying the
1/rms row scale after the GEMM keeps "mathematical equivalence"), linear-layer
grouping (projections that share an input concatenate their A weights) and
low-rank activation checkpointing (the re-forward is confined to the block).
The oracle therefore does NOT fold, group or fuse anything: it normalises
explicitly, runs each pair on its own and derives gradients by the textbook
chain rule.  Checkpoint mode re-runs the block's forward from its saved input
and bottleneck pre-activations, and must give gradients bitwise equal to the
no-checkpoint mode.

Precision: float64 throughout.  Inputs stored in bf16 or fp32 are widened to
float64 exactly.  Matrix products use numpy's ``@`` (a library primitive).

Pins (checked by tests/test_oracle.py against mathematics, not against this
file's own formulas): sigma = identity reduces a pair to the dense product
(B A) v; central finite differences of every gradient on tiny sizes; the folded
forms of the norm (s . (A * g) . x) against explicit RMSNorm; stacked-A GEMMs
against separate ones; SiLU special values; checkpoint == no-checkpoint
gradients bitwise.  No function here is parity unpinned.
"""
from __future__ import annotations

from typing import Callable, Dict, List, Optional, Sequence, Tuple

import numpy as np

F64 = np.float64

__all__ = [
    "to64",
    "silu",
    "silu_grad",
    "identity",
    "identity_grad",
    "rmsnorm",
    "rmsnorm_bwd",
    "lowrank_fwd",
    "lowrank_bwd",
    "mlp_block_fwd",
    "mlp_block_bwd",
    "proj_group_fwd",
    "proj_group_bwd",
    "mse",
    "stack_step",
    "FULL",
    "CKPT",
]

FULL = "full"  # keep every forward intermediate for the backward
CKPT = "ckpt"  # keep only the block input, the bottleneck pre-activations and 1/rms


def to64(a) -> np.ndarray:
    """Widen a torch tensor or array (bf16 / fp32 / fp64) exactly to a float64 ndarray."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor; bf16 -> fp32 is exact, fp32 -> fp64 is exact
        t = a.detach().cpu()
        if str(t.dtype) in ("torch.bfloat16", "torch.float16"):
            t = t.float()
        return t.double().numpy()
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------------------
# Activation: sigma = SiLU(u) = u * logistic(u)  (this library's reading of the
# pages' unnamed bottleneck nonlinearity; it is also the SwiGLU gate).
# ---------------------------------------------------------------------------
def _logistic(u: np.ndarray) -> np.ndarray:
    # 1 / (1 + e^-u), written so that no exp overflows for large |u|.
    out = np.empty_like(u, dtype=F64)
    pos = u >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-u[pos]))
    e = np.exp(u[~pos])
    out[~pos] = e / (1.0 + e)
    return out


def silu(u: np.ndarray) -> np.ndarray:
    """SiLU(u) = u * logistic(u)."""
    return u * _logistic(u)


def silu_grad(u: np.ndarray) -> np.ndarray:
    """d SiLU / du = lam + u * lam * (1 - lam), lam = logistic(u)."""
    lam = _logistic(u)
    return lam + u * lam * (1.0 - lam)


def identity(u: np.ndarray) -> np.ndarray:
    """sigma = identity: the plain SVD-style factorisation W = B A (technical summary §4 lists SVD)."""
    return u


def identity_grad(u: np.ndarray) -> np.ndarray:
    return np.ones_like(u)


ACTS: Dict[str, Tuple[Callable, Callable]] = {
    "silu": (silu, silu_grad),
    "identity": (identity, identity_grad),
}


# ---------------------------------------------------------------------------
# RMSNorm, explicit (technical summary §2.2, Online-RMSNorm, is an exact
# rewrite of this): s_t = (mean_j x_tj^2 + eps)^(-1/2), n_tj = g_j x_tj s_t.
# ---------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> Tuple[np.ndarray, np.ndarray]:
    """Return (n, s): n = g * x * s with the per-row inverse rms s (mean over d, eps inside the root)."""
    ms = np.mean(x * x, axis=1)
    s = 1.0 / np.sqrt(ms + eps)
    n = x * s[:, None] * g[None, :]
    return n, s


def rmsnorm_bwd(x: np.ndarray, g: np.ndarray, s: np.ndarray, dn: np.ndarray):
    """Chain rule through n = g * x * s(x).

    dn/dx_tk = g_k s_t [j == k] + g_j x_tj ds_t/dx_tk with ds_t/dx_tk = -s_t^3 x_tk / d, hence
    dx_tk = s_t g_k dn_tk - (s_t^3 / d) x_tk sum_j g_j dn_tj x_tj and dg_j = sum_t dn_tj x_tj s_t.
    """
    d = x.shape[1]
    gdn = dn * g[None, :]
    proj = np.sum(gdn * x, axis=1)
    dx = s[:, None] * gdn - (s ** 3 / d)[:, None] * x * proj[:, None]
    dg = np.sum(dn * x * s[:, None], axis=0)
    return dx, dg


# ---------------------------------------------------------------------------
# One low-rank pair y = B sigma(A v)  (technical summary §1/§2.1: each linear
# map becomes an r x d_in layer followed by a d_out x r layer).
# ---------------------------------------------------------------------------
def lowrank_fwd(v: np.ndarray, A: np.ndarray, B: np.ndarray, act: str = "silu"):
    """Return (y, u, z): u = v A^T (pre-activation), z = sigma(u), y = z B^T."""
    f, _ = ACTS[act]
    u = v @ A.T
    z = f(u)
    y = z @ B.T
    return y, u, z


def lowrank_bwd(v: np.ndarray, A: np.ndarray, B: np.ndarray, u: np.ndarray, z: np.ndarray,
                dy: np.ndarray, act: str = "silu"):
    """Return (dv, dA, dB) for y = B sigma(A v) given dL/dy."""
    _, fp = ACTS[act]
    dB = dy.T @ z
    dz = dy @ B
    du = dz * fp(u)
    dA = du.T @ v
    dv = du @ A
    return dv, dA, dB


# ---------------------------------------------------------------------------
# Low-rank SwiGLU MLP block (residual):
#   n = RMSNorm(x); a = LR_gate(n); b = LR_up(n); h = SiLU(a) * b; out = x + LR_down(h)
# ---------------------------------------------------------------------------
_MLP_KEYS = ("A_gate", "B_gate", "A_up", "B_up", "A_down", "B_down")


def _mlp_forward_core(x, g, W, eps, act):
    n, s = rmsnorm(x, g, eps)
    a, u_g, z_g = lowrank_fwd(n, W["A_gate"], W["B_gate"], act)
    b, u_u, z_u = lowrank_fwd(n, W["A_up"], W["B_up"], act)
    h = silu(a) * b
    y, u_d, z_d = lowrank_fwd(h, W["A_down"], W["B_down"], act)
    out = x + y
    inter = dict(n=n, s=s, u_gate=u_g, z_gate=z_g, u_up=u_u, z_up=z_u, a=a, b=b, h=h,
                 u_down=u_d, z_down=z_d)
    return out, inter


def mlp_block_fwd(x, g, W: Dict[str, np.ndarray], eps: float = 1e-6, mode: str = FULL,
                  act: str = "silu"):
    """Forward of one block. Returns (out, saved).

    FULL keeps every intermediate.  CKPT keeps only what low-rank activation
    checkpointing keeps (technical summary §2.2): the block input x, the
    bottleneck pre-activations u_gate, u_up, u_down ([T, r] each) and 1/rms s.
    """
    x, g = to64(x), to64(g)
    W = {k: to64(W[k]) for k in _MLP_KEYS}
    out, inter = _mlp_forward_core(x, g, W, eps, act)
    if mode == FULL:
        saved = dict(inter)
        saved["x"] = x
    elif mode == CKPT:
        saved = dict(x=x, s=inter["s"], u_gate=inter["u_gate"], u_up=inter["u_up"],
                     u_down=inter["u_down"])
    else:
        raise ValueError(mode)
    saved["mode"] = mode
    return out, saved


def _mlp_recompute(saved, g, W, act):
    """Re-forward of a checkpointed block from x, s and the [T, r] pre-activations only."""
    f, _ = ACTS[act]
    x, s = saved["x"], saved["s"]
    n = x * s[:, None] * g[None, :]
    z_g = f(saved["u_gate"])
    z_u = f(saved["u_up"])
    a = z_g @ W["B_gate"].T
    b = z_u @ W["B_up"].T
    h = silu(a) * b
    z_d = f(saved["u_down"])
    return dict(n=n, s=s, u_gate=saved["u_gate"], z_gate=z_g, u_up=saved["u_up"], z_up=z_u,
                a=a, b=b, h=h, u_down=saved["u_down"], z_down=z_d, x=x)


def mlp_block_bwd(g, W: Dict[str, np.ndarray], saved, G, eps: float = 1e-6, act: str = "silu"):
    """Backward of one block given dL/dout = G. Returns dict with dx, dg and dA_*/dB_*."""
    g = to64(g)
    W = {k: to64(W[k]) for k in _MLP_KEYS}
    G = to64(G)
    S = saved if saved["mode"] == FULL else _mlp_recompute(saved, g, W, act)
    x = S["x"]
    # out = x + LR_down(h)
    dh, dA_d, dB_d = lowrank_bwd(S["h"], W["A_down"], W["B_down"], S["u_down"], S["z_down"], G, act)
    # h = SiLU(a) * b
    da = dh * S["b"] * silu_grad(S["a"])
    db = dh * silu(S["a"])
    dn_g, dA_g, dB_g = lowrank_bwd(S["n"], W["A_gate"], W["B_gate"], S["u_gate"], S["z_gate"], da, act)
    dn_u, dA_u, dB_u = lowrank_bwd(S["n"], W["A_up"], W["B_up"], S["u_up"], S["z_up"], db, act)
    dx_n, dg = rmsnorm_bwd(x, g, S["s"], dn_g + dn_u)
    return dict(dx=G + dx_n, dg=dg, dA_gate=dA_g, dB_gate=dB_g, dA_up=dA_u, dB_up=dB_u,
                dA_down=dA_d, dB_down=dB_d)


# ---------------------------------------------------------------------------
# Dense (full-rank) SwiGLU MLP block, the map the low-rank block replaces
# (technical summary §1: each dense W is replaced by a pair; the pages compare
# BOOST with full-rank training):
#   n = RMSNorm(x); a = n W_gate^T; b = n W_up^T; h = SiLU(a) * b; out = x + h W_down^T
# ---------------------------------------------------------------------------
_DENSE_KEYS = ("W_gate", "W_up", "W_down")


def dense_mlp_fwd(x, g, W: Dict[str, np.ndarray], eps: float = 1e-6):
    """Forward of the dense block. Returns (out, saved) with every intermediate kept."""
    x, g = to64(x), to64(g)
    W = {k: to64(W[k]) for k in _DENSE_KEYS}
    n, s = rmsnorm(x, g, eps)
    a = n @ W["W_gate"].T
    b = n @ W["W_up"].T
    h = silu(a) * b
    out = x + h @ W["W_down"].T
    return out, dict(x=x, n=n, s=s, a=a, b=b, h=h)


def dense_mlp_bwd(g, W: Dict[str, np.ndarray], saved, G):
    """Backward of the dense block given dL/dout = G. Returns dict with dx, dg, dW_gate, dW_up, dW_down."""
    g = to64(g)
    W = {k: to64(W[k]) for k in _DENSE_KEYS}
    G = to64(G)
    S = saved
    dW_down = G.T @ S["h"]
    dh = G @ W["W_down"]
    da = dh * S["b"] * silu_grad(S["a"])
    db = dh * silu(S["a"])
    dW_gate = da.T @ S["n"]
    dW_up = db.T @ S["n"]
    dn = da @ W["W_gate"] + db @ W["W_up"]
    dx_n, dg = rmsnorm_bwd(S["x"], g, S["s"], dn)
    return dict(dx=G + dx_n, dg=dg, dW_gate=dW_gate, dW_up=dW_up, dW_down=dW_down)


# ---------------------------------------------------------------------------
# Projection group: pairs that read the same input (q/k/v), optionally behind
# one RMSNorm; technical summary §2.2 "linear-layer grouping" concatenates
# their A weights, which is exact, so the oracle runs them one by one.
# ---------------------------------------------------------------------------
def proj_group_fwd(x, g, As: Sequence, Bs: Sequence, eps: float = 1e-6, act: str = "silu"):
    """Return (outs, saved) with outs[i] = LR_i(RMSNorm(x)) (or LR_i(x) when g is None)."""
    x = to64(x)
    g = to64(g) if g is not None else None
    if g is not None:
        v, s = rmsnorm(x, g, eps)
    else:
        v, s = x, None
    outs, us, zs = [], [], []
    for A, B in zip(As, Bs):
        y, u, z = lowrank_fwd(v, to64(A), to64(B), act)
        outs.append(y)
        us.append(u)
        zs.append(z)
    return outs, dict(x=x, v=v, s=s, u=us, z=zs)


def proj_group_bwd(g, As: Sequence, Bs: Sequence, saved, Gs: Sequence, act: str = "silu"):
    """Return dict(dx, dg (None without norm), dA[i], dB[i]) given dL/douts[i] = Gs[i]."""
    g = to64(g) if g is not None else None
    dv = np.zeros_like(saved["v"])
    dAs, dBs = [], []
    for i, (A, B) in enumerate(zip(As, Bs)):
        dvi, dA, dB = lowrank_bwd(saved["v"], to64(A), to64(B), saved["u"][i], saved["z"][i],
                                  to64(Gs[i]), act)
        dv = dv + dvi
        dAs.append(dA)
        dBs.append(dB)
    if g is not None:
        dx, dg = rmsnorm_bwd(saved["x"], g, saved["s"], dv)
    else:
        dx, dg = dv, None
    return dict(dx=dx, dg=dg, dA=dAs, dB=dBs)


# ---------------------------------------------------------------------------
# Loss and the residual stack.
# ---------------------------------------------------------------------------
def mse(y: np.ndarray, t: np.ndarray) -> Tuple[float, np.ndarray]:
    """L = mean over all T*d elements of (y - t)^2 and dL/dy = 2 (y - t) / (T d)."""
    diff = y - t
    n = diff.size
    return float(np.sum(diff * diff) / n), 2.0 * diff / n


def stack_step(x, target, blocks: List[Dict], eps: float = 1e-6, mode: str = CKPT,
               act: str = "silu"):
    """One training step of L residual MLP blocks and an MSE loss: returns (loss, grads per block, dx)."""
    h = to64(x)
    saves = []
    for blk in blocks:
        h, sv = mlp_block_fwd(h, blk["g"], blk, eps, mode, act)
        saves.append(sv)
    loss, dy = mse(h, to64(target))
    grads: List[Dict] = [None] * len(blocks)
    for l in range(len(blocks) - 1, -1, -1):
        gr = mlp_block_bwd(blocks[l]["g"], blocks[l], saves[l], dy, eps, act)
        dy = gr.pop("dx")
        grads[l] = gr
    return loss, grads, dy


def mlp_block_rows(x_rows, g, W, G_rows, eps: float = 1e-6, act: str = "silu"):
    """out and dx of the block for a subset of rows (both are row-local), without weight grads."""
    out, saved = mlp_block_fwd(x_rows, g, W, eps, FULL, act)
    gr = mlp_block_bwd(g, W, saved, G_rows, eps, act)
    return out, gr["dx"]
