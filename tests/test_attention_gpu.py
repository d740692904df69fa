"""Parity of causal multi-head attention (through the C ABI) with the fp64 oracle.

Inputs are seeded host arrays rounded to bf16; the oracle reads them widened to fp64.  The
figures (oracle.compare) are the per-tensor max-relative error (max |gpu - ref| / max |ref|),
the same per row and per column against the row's (column's) own scale, and the element-wise
error above the bf16 floor, each bound 2e-2 as for the other bf16 paths.  The full-size case (8 x 2048 tokens, 32 heads of 128) is checked on
sampled heads: each head's attention and gradients depend on that head's q, k, v, dout only.
"""
import pytest
import torch

import oracle.attention_oracle as A
import oracle.compare as C

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rank_bottleneck_block_gb300 import build

    build.build()
    from rank_bottleneck_block_gb300 import lowrank as L

    L.lib()
    yield


def _inputs(seed, b, s, H, dh):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn(b * s, H * dh, generator=g).to(torch.bfloat16) for _ in range(4)]


def _run(b, s, H, dh, seed):
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import Attention

    q, k, v, dout = _inputs(seed, b, s, H, dh)
    at = Attention(b, s, H, dh, q, k, v)
    at.forward()
    at.backward(dout.cuda())
    torch.cuda.synchronize()
    L.lr_check_device_error()
    return (q, k, v, dout), at


def _head_cols(h, dh):
    return slice(h * dh, (h + 1) * dh)


# s = 2304: rows longer than the register softmax holds, and an odd number of 256-row pairs;
# dh = 384: the half-warp row dot with more than one pass per lane.
@pytest.mark.parametrize("b,s,H,dh", [(2, 256, 2, 128), (1, 512, 3, 128), (1, 256, 1, 256), (1, 2304, 1, 128),
                                      (1, 256, 1, 384)])
def test_attention_matches_oracle(b, s, H, dh):
    (q, k, v, dout), at = _run(b, s, H, dh, seed=31 + s + H)
    q64, k64, v64, d64 = (t.double().numpy() for t in (q, k, v, dout))
    o, saved = A.attention_fwd(q64, k64, v64, b, s, H, dh, at.scale)
    gr = A.attention_bwd(q64, k64, v64, o, saved, d64, b, s, H, dh, at.scale)
    errs = {"o": C.metrics(at.o, o), "dq": C.metrics(at.dq, gr["dq"]), "dk": C.metrics(at.dk, gr["dk"]),
            "dv": C.metrics(at.dv, gr["dv"])}
    lse = at.saved.view(torch.float32)[: b * H * s].reshape(b * H, s)
    errs["lse"] = C.metrics(lse, saved["lse"].reshape(b * H, s))
    C.assert_close(errs, "bf16", f"attention b={b} s={s} H={H} dh={dh}")


def test_attention_causal_and_deterministic():
    """Changing the last quarter of the keys and values leaves the first three quarters of
    the output bit-for-bit unchanged; a repeated step gives identical gradients."""
    b, s, H, dh = 1, 512, 2, 128
    (q, k, v, dout), at = _run(b, s, H, dh, seed=7)
    o1 = at.o.clone()
    grads = [t.clone() for t in (at.dq, at.dk, at.dv)]
    at.backward()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b_) for a, b_ in zip(grads, (at.dq, at.dk, at.dv)))
    at.k[3 * s // 4:] += 1.0
    at.v[3 * s // 4:] -= 1.0
    at.forward()
    torch.cuda.synchronize()
    assert torch.equal(at.o[: 3 * s // 4], o1[: 3 * s // 4])
    assert not torch.equal(at.o[3 * s // 4:], o1[3 * s // 4:])


@pytest.mark.slow
def test_attention_full_size_sampled_heads():
    """8 sequences of 2048 tokens, 32 heads of 128: o, dq, dk, dv of three heads against the
    oracle run on those heads alone."""
    b, s, H, dh = 8, 2048, 32, 128
    (q, k, v, dout), at = _run(b, s, H, dh, seed=3)
    for bi, h in ((0, 0), (3, 17), (7, 31)):
        rows, cols = slice(bi * s, (bi + 1) * s), _head_cols(h, dh)
        sub = [t[rows, cols].double().numpy() for t in (q, k, v, dout)]
        o, saved = A.attention_fwd(sub[0], sub[1], sub[2], 1, s, 1, dh, at.scale)
        gr = A.attention_bwd(sub[0], sub[1], sub[2], o, saved, sub[3], 1, s, 1, dh, at.scale)
        errs = {"o": C.metrics(at.o[rows, cols], o), "dq": C.metrics(at.dq[rows, cols], gr["dq"]),
                "dk": C.metrics(at.dk[rows, cols], gr["dk"]), "dv": C.metrics(at.dv[rows, cols], gr["dv"])}
        C.assert_close(errs, "bf16", f"head {(bi, h)}")
