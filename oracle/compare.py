"""Parity metrics between a computed fp16 C and the oracle's fp16 C (test infrastructure).

The bar for the fused fp16 GEMM: relative Frobenius error <= 1e-3 over the
checked set, and every element within |err| <= 1e-2 * (1 + |ref|).  (The
tutorial page "TileLang: Write, Autotune, and Ship Fused Tensor-Core Kernels
from Python", Numerical validation, uses relative Frobenius <= 2e-2 as its own
check; the bar here is tighter.)
"""
from __future__ import annotations

import numpy as np

REL_FROB_TOL = 1e-3
ELEM_ATOL = 1e-2
ELEM_RTOL = 1e-2


def parity(got, ref):
    """dict with rel_frob, max_abs, worst element ratio, and pass flag."""
    g = np.asarray(got, dtype=np.float16).astype(np.float64)
    r = np.asarray(ref, dtype=np.float16).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    if g.size == 0:
        return {"rel_frob": 0.0, "max_abs": 0.0, "worst_ratio": 0.0, "n": 0, "ok": True}
    finite = np.isfinite(r)
    nonfinite_ok = bool(np.array_equal(np.isnan(g), np.isnan(r)) and
                        np.array_equal(g[np.isinf(r)], r[np.isinf(r)]))
    d = np.abs(g[finite] - r[finite])
    if not np.all(np.isfinite(g[finite])):
        return {"rel_frob": float("inf"), "max_abs": float("inf"), "worst_ratio": float("inf"),
                "n": int(g.size), "ok": False}
    nr = float(np.linalg.norm(r[finite]))
    nd = float(np.linalg.norm(d))
    rel = nd / nr if nr > 0 else nd
    bound = ELEM_ATOL + ELEM_RTOL * np.abs(r[finite])
    worst = float(np.max(d / bound)) if d.size else 0.0
    ok = nonfinite_ok and (rel <= REL_FROB_TOL if nr > 0 else nd <= 1e-6) and worst <= 1.0
    return {"rel_frob": rel, "max_abs": float(d.max()) if d.size else 0.0, "worst_ratio": worst,
            "n": int(g.size), "ok": bool(ok)}
