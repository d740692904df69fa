"""Writes tests/golden/mlp_tiny_f32.json from the fp64 oracle only.

The pages print no worked numeric example, so this fixture is a regression
guard of the oracle itself (its correctness is pinned by tests/test_oracle.py):
a seeded T=4, d=16, f=24, r=4 fp32 block, its output, dx, dg and the sums of
every weight gradient.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle.lowrank_oracle as O  # noqa: E402
from rank_bottleneck_block_gb300 import inputs as I  # noqa: E402

SHAPE = I.MlpShape(T=4, d=16, f=24, r=4, dtype="f32")


def compute():
    c = I.make_mlp_case(SHAPE, seed=0)
    out, saved = O.mlp_block_fwd(c["x"], c["g"], c, SHAPE.eps, O.CKPT)
    gr = O.mlp_block_bwd(c["g"], c, saved, c["G"], SHAPE.eps)
    res = {"out": out.ravel().tolist(), "dx": gr["dx"].ravel().tolist(), "dg": gr["dg"].tolist()}
    for k in ("gate", "up", "down"):
        res[f"sum_dA_{k}"] = float(gr[f"dA_{k}"].sum())
        res[f"sum_dB_{k}"] = float(gr[f"dB_{k}"].sum())
    return res


if __name__ == "__main__":
    res = compute()
    res["_about"] = "oracle output for inputs.make_mlp_case(MlpShape(T=4,d=16,f=24,r=4,f32), seed=0); mode ckpt"
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "mlp_tiny_f32.json"), "w") as fh:
        json.dump(res, fh, indent=1)
