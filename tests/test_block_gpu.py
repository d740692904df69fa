"""Parity of the low-rank transformer block (through the C ABI) with the fp64 oracle.

The block chains the q/k/v group, causal attention, the o-projection with its residual and
the MLP block; the oracle chains its own pieces (pinned on their own and, composed, by finite
differences).  Figures (oracle.compare): per-tensor max-relative error, the same per row and
per column, and the element-wise error above the bf16 floor, each bound 2e-2 (bf16 storage).  At full
width the oracle runs on whole sequences: each sequence's outputs and input gradient depend
only on that sequence.
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


def _run(shape, seed):
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import TransformerBlock

    case = I.make_block_case(shape, seed)
    blk = TransformerBlock(shape, case)
    blk.forward()
    blk.backward()
    torch.cuda.synchronize()
    L.lr_check_device_error()
    return case, blk


def _oracle(case, shape, rows=None):
    W = {k: v.double().numpy() for k, v in case.items() if k not in ("x", "G")}
    x, G = case["x"].double().numpy(), case["G"].double().numpy()
    b = shape.b
    if rows is not None:
        x, G, b = x[rows], G[rows], 1
    scale = shape.dh ** -0.5
    out, saved = A.block_fwd(x, W, b, shape.s, shape.H, shape.dh, scale, shape.eps)
    return out, A.block_bwd(W, saved, G, b, shape.s, shape.H, shape.dh, scale, shape.eps)


@pytest.mark.parametrize("dims", [(2, 256, 2, 128, 344, 32, 48), (1, 512, 3, 128, 264, 24, 40)])
def test_block_matches_oracle(dims):
    from rank_bottleneck_block_gb300 import inputs as I

    shape = I.BlockShape(*dims)
    case, blk = _run(shape, seed=sum(dims))
    out, gr = _oracle(case, shape)
    errs = {"out": C.metrics(blk.out, out), "dx": C.metrics(blk.dx, gr["dx"]),
            "dg_attn": C.metrics(blk.dg_attn, gr["dg_attn"]), "dg_mlp": C.metrics(blk.dg_mlp, gr["dg_mlp"])}
    for n in ("q", "k", "v", "o", "gate", "up", "down"):
        for m in ("A", "B"):
            errs[f"d{m}_{n}"] = C.weight(blk.grads[f"d{m}_{n}"], gr[f"d{m}_{n}"])
    C.assert_close(errs, "bf16", f"block {dims}")


@pytest.mark.slow
def test_block_full_width_sampled_sequences():
    """d 4096 (32 heads of 128), f 11008, ranks 1024, 8 sequences of 2048 tokens: out and dx of
    the first and the last sequence against the oracle run on that sequence alone."""
    from rank_bottleneck_block_gb300 import inputs as I

    shape = I.BLOCK_7B
    case, blk = _run(shape, seed=0)
    for bi in (0, shape.b - 1):
        rows = slice(bi * shape.s, (bi + 1) * shape.s)
        out, gr = _oracle(case, shape, rows)
        errs = {"out": C.metrics(blk.out[rows], out), "dx": C.metrics(blk.dx[rows], gr["dx"])}
        C.assert_close(errs, "bf16", f"sequence {bi}")


def test_block_steps_back_to_back_repeat_bitwise():
    """Three fwd+bwd steps issued without a synchronisation in between finish and reproduce the
    first step's outputs and gradients bit for bit."""
    from rank_bottleneck_block_gb300 import inputs as I
    from rank_bottleneck_block_gb300 import lowrank as L

    shape = I.BlockShape(2, 256, 2, 128, 344, 32, 48)
    _, blk = _run(shape, seed=5)
    ref = [blk.out.clone(), blk.dx.clone()] + [v.clone() for v in blk.grads.values()]
    for _ in range(3):
        blk.step()
    torch.cuda.synchronize()
    L.lr_check_device_error()
    now = [blk.out, blk.dx] + list(blk.grads.values())
    assert all(torch.equal(a, b) for a, b in zip(ref, now))
