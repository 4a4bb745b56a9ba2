"""Helpers shared by the parity tests: running the oracle on seeded inputs and
the tolerance checks.  Tolerances (bf16 inputs; fp64 oracle):
out max-abs <= 1e-2 and rel-L2 <= 5e-3; LSE max-abs <= 1e-3;
dQ, dK, dV rel-L2 <= 1e-2 (rel-L2 = ||x - ref|| / ||ref|| over the compared
tensor)."""
from __future__ import annotations

import numpy as np

OUT_MAX_ABS = 1e-2
OUT_REL_L2 = 5e-3
LSE_MAX_ABS = 1e-3
GRAD_REL_L2 = 1e-2


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(x - ref) / den) if den > 0 else float(np.linalg.norm(x - ref))


def max_abs(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(x - ref).max()) if x.size else 0.0


def check_forward(out, lse, ref_out, ref_lse, what=""):
    errs = {"out_max_abs": max_abs(out, ref_out), "out_rel_l2": rel_l2(out, ref_out),
            "lse_max_abs": max_abs(lse, ref_lse)}
    assert np.isfinite(np.asarray(out, dtype=np.float64)).all(), f"{what}: non-finite out"
    assert errs["out_max_abs"] <= OUT_MAX_ABS, (what, errs)
    assert errs["out_rel_l2"] <= OUT_REL_L2, (what, errs)
    assert errs["lse_max_abs"] <= LSE_MAX_ABS, (what, errs)
    return errs


def check_grads(pairs, what=""):
    errs = {}
    for name, (x, ref) in pairs.items():
        assert np.isfinite(np.asarray(x, dtype=np.float64)).all(), f"{what}: non-finite {name}"
        errs[name] = rel_l2(x, ref)
        assert errs[name] <= GRAD_REL_L2, (what, name, errs)
    return errs
