"""Shared test helpers: geometry conversion and error metrics (no attention math)."""
import numpy as np

from oracle import swa_oracle as orc


def to_problem(geom) -> "orc.Problem":
    d = geom.as_dict() if hasattr(geom, "as_dict") else dict(geom)
    return orc.Problem(**d)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def max_abs(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref)))
