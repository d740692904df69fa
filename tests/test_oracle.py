"""Pins of the fp64 oracle against mathematics (no GPU).

Each check here is fixed by something other than the oracle's own formulas:
closed forms (sigma = identity gives the dense product), central finite
differences, library routines (torch's fp64 rms_norm / silu / autograd), the
exactness claims of the pages' optimisations (BOOST technical summary §2.2:
Online-RMSNorm keeps mathematical equivalence, grouping concatenates A weights,
checkpointed re-forward stays inside the block), and special values.
The mutation tests at the end plant plausible mistakes in the oracle and
check that at least one pin catches each.
"""
import numpy as np
import pytest
import torch

import oracle.lowrank_oracle as O
from rank_bottleneck_block_gb300 import inputs as I


def rng(seed=0):
    return np.random.default_rng(seed)


def tiny_mlp(seed=0, T=4, d=16, f=24, r=4):
    R = rng(seed)
    W = {
        "A_gate": R.normal(0, d ** -0.5, (r, d)),
        "B_gate": R.normal(0, r ** -0.5, (f, r)),
        "A_up": R.normal(0, d ** -0.5, (r, d)),
        "B_up": R.normal(0, r ** -0.5, (f, r)),
        "A_down": R.normal(0, f ** -0.5, (r, f)),
        "B_down": R.normal(0, r ** -0.5, (d, r)),
    }
    x = R.normal(0, 1, (T, d))
    g = 1 + R.normal(0, 0.1, d)
    G = R.normal(0, 1, (T, d))
    return x, g, W, G


def rel(a, b):
    a, b = np.asarray(a), np.asarray(b)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------- activation
def test_silu_special_values():
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert O.silu_grad(np.array([0.0]))[0] == 0.5
    big = np.array([40.0, 1000.0])
    np.testing.assert_allclose(O.silu(big), big, rtol=1e-15)
    np.testing.assert_allclose(O.silu_grad(big), 1.0, rtol=1e-15)
    neg = np.array([-40.0, -1000.0])
    assert np.all(np.abs(O.silu(neg)) < 1e-15)
    assert np.all(np.abs(O.silu_grad(neg)) < 1e-15)
    # SiLU(u) - SiLU(-u) = u (odd part of u * logistic(u) is u/2 each side)
    u = np.linspace(-8, 8, 101)
    np.testing.assert_allclose(O.silu(u) - O.silu(-u), u, atol=1e-14)


def test_silu_matches_library_and_derivative():
    u = np.linspace(-30, 30, 2001)
    ref = torch.nn.functional.silu(torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(O.silu(u), ref, rtol=1e-14, atol=1e-300)
    h = 1e-6
    fd = (O.silu(u + h) - O.silu(u - h)) / (2 * h)
    np.testing.assert_allclose(O.silu_grad(u), fd, atol=1e-8)


# ------------------------------------------------------------------ rmsnorm
def test_rmsnorm_matches_library():
    R = rng(1)
    x = R.normal(0, 1, (7, 33))
    g = 1 + R.normal(0, 0.1, 33)
    n, s = O.rmsnorm(x, g, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(g), eps=1e-6)
    np.testing.assert_allclose(n, ref.numpy(), rtol=1e-14, atol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    R = rng(2)
    x = R.normal(0, 3, (5, 64))
    n, _ = O.rmsnorm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(n * n, axis=1)), 1.0, rtol=1e-14)
    n2, _ = O.rmsnorm(7.5 * x, np.ones(64), 0.0)
    np.testing.assert_allclose(n2, n, rtol=1e-13)


# ------------------------------------------------------- closed-form pins
def test_identity_activation_gives_dense_product():
    """sigma = identity: B (A v) must equal the dense map (B A) v."""
    R = rng(3)
    A = R.normal(0, 1, (5, 13))
    B = R.normal(0, 1, (11, 5))
    v = R.normal(0, 1, (9, 13))
    y, _, _ = O.lowrank_fwd(v, A, B, act="identity")
    W = B @ A
    np.testing.assert_allclose(y, v @ W.T, rtol=1e-12, atol=1e-12)


def test_identity_mlp_matches_dense_swiglu():
    """With identity bottlenecks the block is the dense SwiGLU MLP with W = B A and torch's RMSNorm."""
    x, g, W, _ = tiny_mlp(4)
    out, _ = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL, act="identity")
    n = torch.nn.functional.rms_norm(torch.from_numpy(x), (x.shape[1],), torch.from_numpy(g), eps=1e-6)
    Wg = torch.from_numpy(W["B_gate"] @ W["A_gate"])
    Wu = torch.from_numpy(W["B_up"] @ W["A_up"])
    Wd = torch.from_numpy(W["B_down"] @ W["A_down"])
    hid = torch.nn.functional.silu(n @ Wg.T) * (n @ Wu.T)
    ref = torch.from_numpy(x) + hid @ Wd.T
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_online_rmsnorm_fold_is_exact():
    """Technical summary §2.2 (Online-RMSNorm): s * (x (A*g)^T) == A applied to RMSNorm(x)."""
    R = rng(5)
    T, d, r = 17, 48, 12
    x = R.normal(0, 1, (T, d))
    g = 1 + R.normal(0, 0.1, d)
    A = R.normal(0, d ** -0.5, (r, d))
    n, _ = O.rmsnorm(x, g, 1e-6)
    s = (np.sum(x * x, axis=1) / d + 1e-6) ** -0.5  # sum of squares accumulated alongside the GEMM
    folded = s[:, None] * (x @ (A * g[None, :]).T)
    np.testing.assert_allclose(folded, n @ A.T, rtol=1e-13, atol=1e-14)


def test_grouping_stacked_equals_separate():
    """Technical summary §2.2 (grouping): concatenated A's in one GEMM give each pair's u exactly."""
    R = rng(6)
    x = R.normal(0, 1, (10, 32))
    As = [R.normal(0, 1, (8, 32)) for _ in range(3)]
    Bs = [R.normal(0, 1, (20, 8)) for _ in range(3)]
    outs, saved = O.proj_group_fwd(x, None, As, Bs)
    U = x @ np.concatenate(As, 0).T
    for i in range(3):
        np.testing.assert_allclose(U[:, 8 * i:8 * (i + 1)], saved["u"][i], rtol=1e-14, atol=1e-14)
        np.testing.assert_allclose(outs[i], O.silu(U[:, 8 * i:8 * (i + 1)]) @ Bs[i].T, rtol=1e-13)
    # grouped dx GEMM (K = group * r) equals the sum of the per-pair dx contributions
    Gs = [R.normal(0, 1, (10, 20)) for _ in range(3)]
    gr = O.proj_group_bwd(None, As, Bs, saved, Gs)
    dus = [(Gs[i] @ Bs[i]) * O.silu_grad(saved["u"][i]) for i in range(3)]
    dx_grouped = np.concatenate(dus, 1) @ np.concatenate(As, 0)
    np.testing.assert_allclose(gr["dx"], dx_grouped, rtol=1e-12, atol=1e-12)


def test_mse_closed_form():
    t = rng(7).normal(0, 1, (3, 5))
    L, dy = O.mse(t + 0.25, t)
    assert abs(L - 0.0625) < 1e-15
    np.testing.assert_allclose(dy, 2 * 0.25 / 15, rtol=1e-14)


# ------------------------------------------------------- finite differences
def _fd_check(loss_fn, params, grads, h=1e-6, tol=1e-6):
    """Central differences of loss_fn over every entry of each param; returns worst relative error."""
    worst = 0.0
    for name, p in params.items():
        fd = np.zeros_like(p)
        it = np.nditer(p, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = p[i]
            p[i] = old + h
            lp = loss_fn()
            p[i] = old - h
            lm = loss_fn()
            p[i] = old
            fd[i] = (lp - lm) / (2 * h)
        e = rel(grads[name], fd)
        worst = max(worst, e)
        assert e < tol, f"{name}: finite-difference mismatch {e:.3e}"
    return worst


@pytest.mark.parametrize("act", ["silu", "identity"])
def test_mlp_block_finite_differences(act):
    x, g, W, G = tiny_mlp(8)

    def loss():
        out, _ = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL, act)
        return float(np.sum(out * G))

    _, saved = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL, act)
    gr = O.mlp_block_bwd(g, W, saved, G, 1e-6, act)
    params = {"x": x, "g": g, **W}
    grads = {"x": gr["dx"], "g": gr["dg"]}
    for k in ("gate", "up", "down"):
        grads[f"A_{k}"] = gr[f"dA_{k}"]
        grads[f"B_{k}"] = gr[f"dB_{k}"]
    _fd_check(loss, params, grads)


@pytest.mark.parametrize("norm", [True, False])
def test_proj_group_finite_differences(norm):
    R = rng(9)
    T, d, dout, r = 5, 16, 12, 4
    x = R.normal(0, 1, (T, d))
    g = 1 + R.normal(0, 0.1, d) if norm else None
    As = [R.normal(0, d ** -0.5, (r, d)) for _ in range(3)]
    Bs = [R.normal(0, r ** -0.5, (dout, r)) for _ in range(3)]
    Gs = [R.normal(0, 1, (T, dout)) for _ in range(3)]

    def loss():
        outs, _ = O.proj_group_fwd(x, g, As, Bs)
        return float(sum(np.sum(o * Gi) for o, Gi in zip(outs, Gs)))

    _, saved = O.proj_group_fwd(x, g, As, Bs)
    gr = O.proj_group_bwd(g, As, Bs, saved, Gs)
    params = {"x": x}
    grads = {"x": gr["dx"]}
    if norm:
        params["g"], grads["g"] = g, gr["dg"]
    for i in range(3):
        params[f"A{i}"], grads[f"A{i}"] = As[i], gr["dA"][i]
        params[f"B{i}"], grads[f"B{i}"] = Bs[i], gr["dB"][i]
    _fd_check(loss, params, grads)


def test_stack_finite_differences_and_checkpoint():
    x, _, _, _ = tiny_mlp(10)
    blocks = []
    for l in range(2):
        _, g, W, _ = tiny_mlp(11 + l)
        blocks.append(dict(g=g, **W))
    target = rng(12).normal(0, 1, x.shape)

    def loss():
        return O.stack_step(x, target, blocks, 1e-6, O.FULL)[0]

    L, grads, dx = O.stack_step(x, target, blocks, 1e-6, O.FULL)
    params, gmap = {"x": x}, {"x": dx}
    for l, blk in enumerate(blocks):
        params[f"g{l}"], gmap[f"g{l}"] = blk["g"], grads[l]["dg"]
        for k in ("gate", "up", "down"):
            for m in ("A", "B"):
                params[f"{m}_{k}{l}"] = blk[f"{m}_{k}"]
                gmap[f"{m}_{k}{l}"] = grads[l][f"d{m}_{k}"]
    _fd_check(loss, params, gmap)
    # low-rank activation checkpointing: the re-forward reproduces the forward exactly
    Lc, gc, dxc = O.stack_step(x, target, blocks, 1e-6, O.CKPT)
    assert Lc == L
    assert np.array_equal(dxc, dx)
    for a, b in zip(grads, gc):
        for k in a:
            assert np.array_equal(a[k], b[k]), k


def test_checkpoint_bitwise_mlp():
    x, g, W, G = tiny_mlp(13, T=32, d=64, f=96, r=16)
    outf, sf = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL)
    outc, sc = O.mlp_block_fwd(x, g, W, 1e-6, O.CKPT)
    assert np.array_equal(outf, outc)
    assert set(sc) == {"x", "s", "u_gate", "u_up", "u_down", "mode"}
    gf = O.mlp_block_bwd(g, W, sf, G)
    gc = O.mlp_block_bwd(g, W, sc, G)
    for k in gf:
        assert np.array_equal(gf[k], gc[k]), k


def test_backward_matches_autograd_moderate_size():
    """torch fp64 autograd on the definition, at sizes finite differences would be slow for."""
    x, g, W, G = tiny_mlp(14, T=64, d=96, f=160, r=24)
    _, saved = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL)
    gr = O.mlp_block_bwd(g, W, saved, G)
    tx = torch.from_numpy(x.copy()).requires_grad_()
    tg = torch.from_numpy(g.copy()).requires_grad_()
    tW = {k: torch.from_numpy(v.copy()).requires_grad_() for k, v in W.items()}
    F = torch.nn.functional
    n = F.rms_norm(tx, (x.shape[1],), tg, eps=1e-6)
    lr = lambda v, k: F.silu(v @ tW[f"A_{k}"].T) @ tW[f"B_{k}"].T  # noqa: E731
    out = tx + lr(F.silu(lr(n, "gate")) * lr(n, "up"), "down")
    (out * torch.from_numpy(G)).sum().backward()
    assert rel(gr["dx"], tx.grad.numpy()) < 1e-12
    assert rel(gr["dg"], tg.grad.numpy()) < 1e-12
    for k in ("gate", "up", "down"):
        assert rel(gr[f"dA_{k}"], tW[f"A_{k}"].grad.numpy()) < 1e-12
        assert rel(gr[f"dB_{k}"], tW[f"B_{k}"].grad.numpy()) < 1e-12


# ------------------------------------------------------- dense (full-rank) block
def tiny_dense(seed, T=5, d=16, f=24):
    R = rng(seed)
    x = R.standard_normal((T, d))
    g = 1.0 + 0.1 * R.standard_normal(d)
    W = {"W_gate": R.standard_normal((f, d)) / np.sqrt(d), "W_up": R.standard_normal((f, d)) / np.sqrt(d),
         "W_down": R.standard_normal((d, f)) / np.sqrt(f)}
    G = R.standard_normal((T, d))
    return x, g, W, G


def test_dense_block_finite_differences():
    x, g, W, G = tiny_dense(31)

    def loss():
        out, _ = O.dense_mlp_fwd(x, g, W, 1e-6)
        return float(np.sum(out * G))

    _, saved = O.dense_mlp_fwd(x, g, W, 1e-6)
    gr = O.dense_mlp_bwd(g, W, saved, G)
    _fd_check(loss, {"x": x, "g": g, **W}, {"x": gr["dx"], "g": gr["dg"], "W_gate": gr["dW_gate"],
                                            "W_up": gr["dW_up"], "W_down": gr["dW_down"]})


def test_dense_block_is_the_lowrank_block_with_identity_factors():
    """r = d, A_gate = A_up = I, B = W, A_down = W_down, B_down = I and sigma = identity turn the
    low-rank block into the dense one: outputs and every gradient agree."""
    x, g, W, G = tiny_dense(32, T=6, d=16, f=24)
    d = x.shape[1]
    I_d = np.eye(d)
    L = {"A_gate": I_d, "B_gate": W["W_gate"], "A_up": I_d, "B_up": W["W_up"], "A_down": W["W_down"],
         "B_down": I_d}
    out_l, sv_l = O.mlp_block_fwd(x, g, L, 1e-6, O.FULL, act="identity")
    gr_l = O.mlp_block_bwd(g, L, sv_l, G, 1e-6, act="identity")
    out_d, sv_d = O.dense_mlp_fwd(x, g, W, 1e-6)
    gr_d = O.dense_mlp_bwd(g, W, sv_d, G)
    assert rel(out_d, out_l) < 1e-13
    assert rel(gr_d["dx"], gr_l["dx"]) < 1e-12
    assert rel(gr_d["dg"], gr_l["dg"]) < 1e-12
    assert rel(gr_d["dW_gate"], gr_l["dB_gate"]) < 1e-12
    assert rel(gr_d["dW_up"], gr_l["dB_up"]) < 1e-12
    assert rel(gr_d["dW_down"], gr_l["dA_down"]) < 1e-12


def test_dense_block_matches_autograd():
    x, g, W, G = tiny_dense(33, T=48, d=64, f=96)
    _, saved = O.dense_mlp_fwd(x, g, W, 1e-6)
    gr = O.dense_mlp_bwd(g, W, saved, G)
    tx = torch.from_numpy(x.copy()).requires_grad_()
    tg = torch.from_numpy(g.copy()).requires_grad_()
    tW = {k: torch.from_numpy(v.copy()).requires_grad_() for k, v in W.items()}
    F = torch.nn.functional
    n = F.rms_norm(tx, (x.shape[1],), tg, eps=1e-6)
    out = tx + (F.silu(n @ tW["W_gate"].T) * (n @ tW["W_up"].T)) @ tW["W_down"].T
    (out * torch.from_numpy(G)).sum().backward()
    assert rel(gr["dx"], tx.grad.numpy()) < 1e-12
    assert rel(gr["dg"], tg.grad.numpy()) < 1e-12
    for k in W:
        assert rel(gr[f"d{k}"], tW[k].grad.numpy()) < 1e-12, k


def test_folded_backward_forms_match_explicit():
    """The folded forms a fused implementation uses (gain inside A, 1/rms as a row scale,
    rho = sum_i du_i u_i) agree with the oracle's explicit RMSNorm backward."""
    x, g, W, G = tiny_mlp(15, T=32, d=64, f=96, r=16)
    _, S = O.mlp_block_fwd(x, g, W, 1e-6, O.FULL)
    gr = O.mlp_block_bwd(g, W, S, G)
    d = x.shape[1]
    Ast = np.concatenate([W["A_gate"], W["A_up"]], 0)
    Af = Ast * g[None, :]
    s = S["s"]
    u = np.concatenate([S["u_gate"], S["u_up"]], 1)
    # recover du from the oracle's own pieces via the definition of the down / SwiGLU chain
    dh = ((G @ W["B_down"]) * O.silu_grad(S["u_down"])) @ W["A_down"]
    da = dh * S["b"] * O.silu_grad(S["a"])
    db = dh * O.silu(S["a"])
    du = np.concatenate([(da @ W["B_gate"]) * O.silu_grad(S["u_gate"]),
                         (db @ W["B_up"]) * O.silu_grad(S["u_up"])], 1)
    du_s = s[:, None] * du
    rho = np.sum(du * u, axis=1)
    dx = G + du_s @ Af - (s * s / d * rho)[:, None] * x
    dAf = du_s.T @ x
    assert rel(dx, gr["dx"]) < 1e-12
    assert rel(dAf * g[None, :], np.concatenate([gr["dA_gate"], gr["dA_up"]], 0)) < 1e-12
    assert rel(np.sum(dAf * Ast, axis=0), gr["dg"]) < 1e-12


def test_inputs_are_seeded_and_shaped():
    shape = I.MlpShape(T=8, d=16, f=24, r=4, dtype="bf16")
    a = I.make_mlp_case(shape, seed=0)
    b = I.make_mlp_case(shape, seed=0)
    for k in a:
        assert torch.equal(a[k], b[k])
        assert a[k].dtype == torch.bfloat16
    assert a["A_gate"].shape == (4, 16) and a["B_down"].shape == (16, 4)
    assert len(I.sweep_shapes()) == 144


# ---------------------------------------------------------- mutation tests
def _mutated(monkeypatch, name, fn):
    monkeypatch.setattr(O, name, fn)


def _fd_fails(act="silu"):
    try:
        test_mlp_block_finite_differences(act)
    except AssertionError:
        return True
    return False


def test_pins_catch_dropped_silu_term(monkeypatch):
    orig = O._logistic
    _mutated(monkeypatch, "silu_grad", lambda u: orig(u))
    assert _fd_fails()


def test_pins_catch_dropped_rmsnorm_projection_term(monkeypatch):
    def bad(x, g, s, dn):
        return s[:, None] * dn * g[None, :], np.sum(dn * x * s[:, None], axis=0)

    _mutated(monkeypatch, "rmsnorm_bwd", bad)
    assert _fd_fails("identity")


def test_pins_catch_wrong_rms_denominator(monkeypatch):
    def bad(x, g, eps):
        s = 1.0 / np.sqrt(np.sum(x * x, axis=1) / (x.shape[1] - 1) + eps)
        return x * s[:, None] * g[None, :], s

    _mutated(monkeypatch, "rmsnorm", bad)
    with pytest.raises(AssertionError):
        test_rmsnorm_matches_library()


def test_pins_catch_swapped_lowrank_factors(monkeypatch):
    def bad(v, A, B, u, z, dy, act="silu"):
        _, fp = O.ACTS[act]
        dz = dy @ B
        du = dz * fp(u)
        return du @ A, du.T @ v, z.T @ dy  # dB transposed-and-swapped

    _mutated(monkeypatch, "lowrank_bwd", bad)
    with pytest.raises(Exception):
        test_mlp_block_finite_differences("silu")


def test_golden_regression():
    """The oracle reproduces the committed fixture written by tests/golden/make_golden.py."""
    import json
    import os

    import importlib.util

    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    with open(os.path.join(here, "mlp_tiny_f32.json")) as fh:
        ref = json.load(fh)
    got = mg.compute()
    for k, v in got.items():
        np.testing.assert_allclose(np.asarray(v), np.asarray(ref[k]), rtol=1e-12, atol=1e-12)
