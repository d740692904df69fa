"""Pins of the attention oracle against definitions it does not share code with.

Brute force (explicit loops over tokens and keys on tiny sizes), central finite differences
of every gradient, causality, and two closed-form special cases.
"""
import math

import numpy as np
import pytest

import oracle.attention_oracle as A


def _rand(seed, b, s, H, dh):
    R = np.random.default_rng(seed)
    return [R.standard_normal((b * s, H * dh)) for _ in range(3)]


def _brute(q, k, v, b, s, H, dh, scale):
    """Each output element from its definition: a loop over keys with a max-shifted softmax."""
    o = np.zeros((b * s, H * dh))
    for bi in range(b):
        for h in range(H):
            cols = slice(h * dh, (h + 1) * dh)
            for i in range(s):
                qi = q[bi * s + i, cols]
                logits = [scale * float(np.dot(qi, k[bi * s + j, cols])) for j in range(i + 1)]
                mx = max(logits)
                w = [math.exp(x - mx) for x in logits]
                tot = sum(w)
                for j in range(i + 1):
                    o[bi * s + i, cols] += (w[j] / tot) * v[bi * s + j, cols]
    return o


def test_forward_matches_brute_force():
    b, s, H, dh = 2, 5, 3, 4
    q, k, v = _rand(0, b, s, H, dh)
    o, saved = A.attention_fwd(q, k, v, b, s, H, dh, 0.7)
    np.testing.assert_allclose(o, _brute(q, k, v, b, s, H, dh, 0.7), rtol=1e-12, atol=1e-12)
    assert saved["lse"].shape == (b, H, s)


def test_lse_is_the_row_log_partition():
    b, s, H, dh = 1, 6, 2, 3
    q, k, v = _rand(1, b, s, H, dh)
    _, saved = A.attention_fwd(q, k, v, b, s, H, dh, 0.5)
    Q, K = A.heads(q, b, s, H, dh), A.heads(k, b, s, H, dh)
    for h in range(H):
        for i in range(s):
            logits = [0.5 * float(np.dot(Q[0, h, i], K[0, h, j])) for j in range(i + 1)]
            assert saved["lse"][0, h, i] == pytest.approx(math.log(sum(math.exp(x) for x in logits)), rel=1e-12)


def test_first_token_returns_its_value_and_zero_queries_average():
    b, s, H, dh = 2, 7, 2, 5
    q, k, v = _rand(2, b, s, H, dh)
    o, _ = A.attention_fwd(q, k, v, b, s, H, dh, 1.0)
    for bi in range(b):
        np.testing.assert_allclose(o[bi * s], v[bi * s], rtol=1e-12)  # only key 0 is visible
    o0, _ = A.attention_fwd(np.zeros_like(q), k, v, b, s, H, dh, 1.0)
    for bi in range(b):
        for i in range(s):  # equal logits: the mean of the visible values
            np.testing.assert_allclose(o0[bi * s + i], v[bi * s:bi * s + i + 1].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_causality():
    b, s, H, dh = 1, 8, 2, 4
    q, k, v = _rand(3, b, s, H, dh)
    o, _ = A.attention_fwd(q, k, v, b, s, H, dh, 0.8)
    k2, v2 = k.copy(), v.copy()
    k2[5:] += 3.0
    v2[5:] -= 2.0
    o2, _ = A.attention_fwd(q, k2, v2, b, s, H, dh, 0.8)
    np.testing.assert_array_equal(o[:5], o2[:5])
    assert not np.allclose(o[5:], o2[5:])


def test_gradients_match_finite_differences():
    b, s, H, dh, scale = 1, 4, 2, 3, 0.6
    q, k, v = _rand(4, b, s, H, dh)
    G = np.random.default_rng(5).standard_normal((b * s, H * dh))
    o, saved = A.attention_fwd(q, k, v, b, s, H, dh, scale)
    gr = A.attention_bwd(q, k, v, o, saved, G, b, s, H, dh, scale)

    def loss(qq, kk, vv):
        return float(np.sum(A.attention_fwd(qq, kk, vv, b, s, H, dh, scale)[0] * G))

    h = 1e-6
    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        num = np.zeros_like(q)
        for i in range(q.shape[0]):
            for j in range(q.shape[1]):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[idx][i, j] += h
                args_m[idx][i, j] -= h
                num[i, j] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(gr[name], num, rtol=1e-6, atol=1e-8, err_msg=name)


def _tiny_block(seed=9, b=1, s=3, H=2, dh=2, f=6, r=2):
    R = np.random.default_rng(seed)
    d = H * dh
    W = {"g_attn": 1 + 0.1 * R.standard_normal(d), "g_mlp": 1 + 0.1 * R.standard_normal(d)}
    for n in "qkvo":
        W[f"A_{n}"] = R.standard_normal((r, d)) / np.sqrt(d)
        W[f"B_{n}"] = R.standard_normal((d, r)) / np.sqrt(r)
    for n, (din, dout) in (("gate", (d, f)), ("up", (d, f)), ("down", (f, d))):
        W[f"A_{n}"] = R.standard_normal((r, din)) / np.sqrt(din)
        W[f"B_{n}"] = R.standard_normal((dout, r)) / np.sqrt(r)
    x = R.standard_normal((b * s, d))
    G = R.standard_normal((b * s, d))
    return W, x, G, (b, s, H, dh)


def test_block_gradients_match_finite_differences():
    """The whole transformer block (q/k/v group, attention, o-projection and its residual,
    MLP block): every gradient against central differences of sum(out * G)."""
    W, x, G, shp = _tiny_block()
    scale = 0.7
    out, saved = A.block_fwd(x, W, *shp, scale)
    gr = A.block_bwd(W, saved, G, *shp, scale)

    def loss(xx, WW):
        return float(np.sum(A.block_fwd(xx, WW, *shp, scale)[0] * G))

    h = 1e-6

    def fd(get, shape):
        num = np.zeros(shape)
        for idx in np.ndindex(*shape):
            xp, Wp = x.copy(), {k: v.copy() for k, v in W.items()}
            xm, Wm = x.copy(), {k: v.copy() for k, v in W.items()}
            get(xp, Wp)[idx] += h
            get(xm, Wm)[idx] -= h
            num[idx] = (loss(xp, Wp) - loss(xm, Wm)) / (2 * h)
        return num

    np.testing.assert_allclose(gr["dx"], fd(lambda xx, WW: xx, x.shape), rtol=1e-6, atol=1e-8)
    for key, g in (("g_attn", "dg_attn"), ("g_mlp", "dg_mlp")):
        np.testing.assert_allclose(gr[g], fd(lambda xx, WW, key=key: WW[key], W[key].shape), rtol=1e-6, atol=1e-8)
    for n in ("q", "k", "v", "o", "gate", "down"):
        for m in ("A", "B"):
            key = f"{m}_{n}"
            np.testing.assert_allclose(gr[f"d{key}"], fd(lambda xx, WW, key=key: WW[key], W[key].shape),
                                       rtol=1e-6, atol=1e-8, err_msg=key)
