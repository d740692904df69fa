"""The comparison figures of oracle.compare catch the mistakes the max-relative error lets through.

CPU only.  Each case plants a mistake in a copy of a reference tensor (never in the library) and
checks which figure flags it.
"""
import numpy as np

import oracle.compare as C


def _weight_grad(rng, units=40, feats=136, tokens=200):
    du = rng.standard_normal((tokens, units))
    du[:, 7] *= 1e-3  # a rarely active unit: its row of the gradient is 1e-3 of the others
    x = rng.standard_normal((tokens, feats))
    return du.T @ x


def test_a_wrong_small_row_passes_maxrel_but_not_the_row_figure():
    rng = np.random.default_rng(0)
    ref = _weight_grad(rng)
    bad = ref.copy()
    bad[7] *= 1.5  # the small unit's gradient 50% off
    m = C.weight(bad, ref, "bf16", tokens=200)
    assert m["maxrel"] <= C.TOL["bf16"]  # invisible next to the tensor's largest values
    assert "row" in C.failures({"dA": m}, "bf16")["dA"][0]


def test_a_small_wrong_column_is_caught_by_the_column_figure():
    rng = np.random.default_rng(1)
    ref = _weight_grad(rng).T.copy()  # [feats, units]: the small unit is a column now
    bad = ref.copy()
    bad[:, 7] = -bad[:, 7]  # wrong sign on a small column
    m = C.weight(bad, ref, "bf16", tokens=200)
    assert m["maxrel"] <= C.TOL["bf16"]
    assert C.failures({"dB": m}, "bf16")["dB"][0] == "col"


def test_rounding_level_errors_pass_every_figure():
    rng = np.random.default_rng(2)
    ref = _weight_grad(rng)
    noisy = ref + 2e-3 * np.abs(ref).max() * rng.standard_normal(ref.shape) * 0.1
    noisy[7] = ref[7] * (1 + 2e-3 * rng.standard_normal(ref.shape[1]))  # the small row at its own scale
    assert not C.failures({"dA": C.weight(noisy, ref, "bf16", tokens=200)}, "bf16")


def test_dg_element_against_its_terms():
    """A dg entry that is small because its terms cancel may carry the terms' rounding error, but
    a wrong small entry whose terms are small too is flagged."""
    rng = np.random.default_rng(3)
    r, d = 32, 64
    A = rng.standard_normal((r, d))
    g = 1 + 0.1 * rng.standard_normal(d)
    dA = rng.standard_normal((r, d))
    dA[:, 5] *= 1e-4  # feature 5: every term small
    ref = (dA * A).sum(axis=0) / g
    scale = C.dg_scale([dA], [A], g)
    ok = ref + 1e-3 * scale * rng.standard_normal(d)  # rounding of each entry's own terms
    assert not C.failures({"dg": C.metrics(ok, ref, "bf16", scale=scale)}, "bf16")
    bad = ref.copy()
    bad[5] *= 2.0
    m = C.metrics(bad, ref, "bf16", scale=scale)
    assert m["maxrel"] <= C.TOL["bf16"]
    assert C.failures({"dg": m}, "bf16")["dg"][0] == "elem"
    assert m["worst"][0] == (5,)


def test_non_finite_values_fail():
    ref = np.ones((4, 4))
    bad = ref.copy()
    bad[1, 2] = np.nan
    try:
        C.metrics(bad, ref)
    except AssertionError:
        return
    raise AssertionError("a NaN passed")
