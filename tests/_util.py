"""Shared helpers for the GPU tests: tolerance checks against the fp64 oracle."""

import numpy as np

# Per-element bound |gpu - ref| <= ATOL + RTOL |ref| and a relative Frobenius
# bound over the evaluated set.
ATOL = 1e-2
RTOL = 1e-2
FRO = 5e-3

# (what, worst element as a fraction of its bound, relative Frobenius) of every
# check in this session, printed in the terminal summary.
RECORD = []


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    worst = float((err / (ATOL + RTOL * np.abs(ref))).max()) if err.size else 0.0
    den = np.linalg.norm(ref)
    fro = float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got - ref))
    return worst, fro, float(err.max()) if err.size else 0.0


def assert_close(got, ref, what="", fro_bound=FRO):
    worst, fro, emax = errors(got, ref)
    RECORD.append((what, worst, fro))
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite values"
    assert worst <= 1.0 and fro <= fro_bound, (
        f"{what}: worst element at {worst:.3f} of the per-element bound, rel Frobenius {fro:.3e} "
        f"(bound {fro_bound:.1e}), max abs err {emax:.3e}")
    return worst, fro
