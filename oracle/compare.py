"""Error figures for comparing a computed tensor with the oracle's.

TEST INFRASTRUCTURE ONLY (like the rest of ``oracle/``): used by ``tests/`` and
``__graft_entry__.smoke()``; nothing on the product path imports it.  It holds
no arithmetic of the method, only the comparison.

Figures per tensor, each bounded in ``failures``:

* ``maxrel`` = max_i |g_i - r_i| / max_i |r_i|, the per-tensor max-relative
  error the tolerances are stated in (2e-2 for bf16 storage, 1e-5 for fp32);
* ``row`` (and ``col`` where asked): for every row (column),
  max_j |g - r| / max(max_j |r|, ROW_FLOOR * max |r|).  A token row of an
  activation, or a unit's row / an input feature's column of a weight gradient,
  is judged against its own scale, so a row that is small next to the tensor's
  largest one (a rarely active unit, an eps-dominated input row next to rows of
  magnitude 1e3) cannot be badly wrong and still pass.  The errors of a
  GEMM-shaped result scale with that row's own operands, so the figure stays at
  the tensor's level; its bound is ROW_TOL_FACTOR times the tolerance because a
  row's largest value estimates its scale from few samples (a weight-gradient
  row of r = 40 columns); lines of fewer than MIN_LINE values are not judged
  this way (their largest value is no estimate of their scale: a row of 24
  values reached 3.1x the tolerance on a correct result);
* ``elem`` = max_i |g_i - r_i| / max(|r_i|, scale_i), where ``scale`` is the
  magnitude of the terms the element sums (given by the caller, e.g. for dg:
  sum_i |dA_ij A_ij| / |g_j|).  An element that is small only because its terms
  cancel keeps the absolute rounding error of those terms, so without the
  terms' magnitude an element-wise relative error has no bound for rounded
  arithmetic; against it, the element-wise error is bounded by the tolerance.
  Without a ``scale`` the figure uses ELEM_FLOOR * max |r| and is reported, not
  bounded: measured on this library's bf16 path, the largest errors sit at
  about 0.4-0.7% of a tensor's largest value irrespective of the element's own
  size (they come from the bf16 rounding of stored intermediates), so a floor
  below ~0.4 of the largest value cannot hold at the 2e-2 tolerance.

``worst`` reports the element with the largest ``elem`` ratio (index, computed
value, oracle value).
"""
from __future__ import annotations

from typing import Dict, Optional, Tuple

import numpy as np

ROW_FLOOR = 1e-3
ROW_TOL_FACTOR = 3.0
MIN_LINE = 32
ELEM_FLOOR = {"bf16": 1e-3, "f32": 1e-3}
TOL = {"bf16": 2e-2, "f32": 1e-5}


def as64(t) -> np.ndarray:
    """Widen a torch tensor (any device, bf16 / fp32) or array to a float64 ndarray."""
    if hasattr(t, "detach"):
        t = t.detach()
        if t.is_cuda:
            t = t.cpu()
        return t.float().double().numpy()
    return np.asarray(t, dtype=np.float64)


def metrics(gpu, ref, dtype: str = "bf16", scale: Optional[np.ndarray] = None, rows: bool = True,
            cols: bool = False) -> Dict[str, object]:
    """The figures (and the worst element) of a computed tensor against the oracle's.

    rows / cols: compute the per-row / per-column figure (2-D tensors); scale: the magnitude of
    each element's terms (same shape), which makes ``elem`` a bounded figure."""
    g, r = as64(gpu), as64(ref)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), "non-finite values in the computed tensor"
    diff = np.abs(g - r)
    ar = np.abs(r)
    M = float(ar.max()) if ar.size else 0.0
    if M == 0.0:  # an all-zero reference: every figure is the absolute error
        M = 1.0
    out: Dict[str, object] = {"maxrel": float(diff.max() / M) if diff.size else 0.0}
    if scale is not None:
        sc = np.asarray(scale, dtype=np.float64)
        assert sc.shape == r.shape, (sc.shape, r.shape)
        den = np.maximum(ar, sc)
        den = np.where(den > 0, den, 1.0)
        out["elem_bounded"] = True
    else:
        den = np.maximum(ar, ELEM_FLOOR[dtype] * M)
    ratio = diff / den
    if ratio.size:
        i = int(np.argmax(ratio))
        out["elem"] = float(ratio.flat[i])
        out["worst"] = (tuple(int(v) for v in np.unravel_index(i, ratio.shape)), float(g.flat[i]), float(r.flat[i]))
    if g.ndim == 2 and g.size:
        # a line (row or column) of fewer than MIN_LINE values estimates its scale from too few samples
        if rows and g.shape[1] >= MIN_LINE:
            out["row"] = float(np.max(diff.max(axis=1) / np.maximum(ar.max(axis=1), ROW_FLOOR * M)))
        if cols and g.shape[0] >= MIN_LINE:
            out["col"] = float(np.max(diff.max(axis=0) / np.maximum(ar.max(axis=0), ROW_FLOOR * M)))
    return out


MIN_TOKENS_FOR_ROWS = 16


def weight(gpu, ref, dtype: str = "bf16", tokens: int = MIN_TOKENS_FOR_ROWS) -> Dict[str, object]:
    """A weight gradient (a sum over `tokens` rows of outer products): rows (units or output features)
    and columns both judged at their own scale.  Below MIN_TOKENS_FOR_ROWS tokens a row is close to
    one outer product of single elements, so its scale is one element's and the row figure would be
    an unbounded element-wise error: only the max-relative error is taken."""
    many = tokens >= MIN_TOKENS_FOR_ROWS
    return metrics(gpu, ref, dtype, rows=many, cols=many)


def dg_scale(dA_list, A_list, g) -> np.ndarray:
    """Magnitude of the terms of dg_j = sum_i dA'_ij A_ij over the stacked normed A's, dA' = dA / g_j
    (the folded form of the RMSNorm gain gradient): sum_i |dA_ij A_ij| / |g_j|."""
    g = as64(g)
    tot = np.zeros_like(g)
    for dA, A in zip(dA_list, A_list):
        tot += np.abs(as64(dA) * as64(A)).sum(axis=0)
    return tot / np.abs(g)


def failures(errs: Dict[str, Dict[str, object]], dtype: str) -> Dict[str, Tuple[str, float]]:
    """The bounded figures of `errs` (name -> metrics) above their bound: name -> (figure, value)."""
    tol = TOL[dtype]
    bad = {}
    for name, m in errs.items():
        checks = [("maxrel", tol), ("row", ROW_TOL_FACTOR * tol), ("col", ROW_TOL_FACTOR * tol)]
        if m.get("elem_bounded"):
            checks.append(("elem", tol))
        for key, bound in checks:
            if key in m and not m[key] <= bound:
                bad[name] = (key, m[key])
                break
    return bad


def summary(errs: Dict[str, Dict[str, object]]) -> str:
    """One line per tensor: its figures and worst element."""
    lines = []
    for name, m in errs.items():
        figs = " ".join(f"{k}={m[k]:.2e}" for k in ("maxrel", "row", "col", "elem") if k in m)
        lines.append(f"{name}: {figs} worst={m.get('worst')}")
    return "\n".join(lines)


def assert_close(errs: Dict[str, Dict[str, object]], dtype: str, what: str = "") -> None:
    bad = failures(errs, dtype)
    assert not bad, f"{what}: {bad}\n{summary(errs)}"
