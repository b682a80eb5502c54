"""Shared test helpers: geometry conversion, error metrics and the parity gates
(no attention math).

The gates (bf16 or fp16 inputs, fp32 accumulation):
- out: relative L2 <= 5e-3; dq / dk / dv: relative L2 <= 1e-2;
- every element of out / dq / dk / dv: |got - ref| <= 2e-2 + half an ulp of
  the output type at |ref|.  The result is stored in bf16 (or fp16), and
  rounding the exact value to that type alone moves it by up to half an ulp
  (2^-6 on [4, 8) in bf16), so the flat 2e-2 bound is kept and only the
  storage rounding of the output itself is added.  fp32 outputs have no such
  rounding: there the bound is the flat 2e-2;
- softmax_max / softmax_sum: relative error <= 1e-3 wherever |ref| >= 1e-3,
  and an absolute error <= 1e-6 (1e-3 of 1e-3) below that; rows with no
  visible key must be -inf / 0 on both sides.

Every comparison is recorded (case, tensor, max |got - ref|, worst margin to
the gate, relative L2) and printed at the end of the session, so each run
leaves the max-abs error it reached per tensor and per case.
"""
import numpy as np

from oracle import swa_oracle as orc

TOL_OUT = 5e-3
TOL_GRAD = 1e-2
TOL_ABS = 2e-2
TOL_STAT = 1e-3
STAT_FLOOR = 1e-3

# (case, tensor, max_abs, excess, rel_l2) of every check this session
REPORT = []


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


def half_ulp(ref, dtype: str) -> np.ndarray:
    """Half a unit in the last place of `dtype` ("bf16", "fp16", "fp32") at
    |ref|: the most that rounding the exact value to the stored type moves it.
    fp32 outputs are compared without it (0)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    if dtype == "fp32":
        return np.zeros_like(a)
    frac_bits, emin = {"bf16": (7, -126), "fp16": (10, -14)}[dtype]
    _, e2 = np.frexp(a)  # a = m * 2**e2, m in [0.5, 1): the binade is [2**(e2-1), 2**e2)
    e = np.maximum(e2 - 1, emin)
    return np.where(a > 0.0, np.ldexp(0.5, (e - frac_bits).astype(np.int64)), 0.0)


def elem_excess(got, ref, dtype: str = "bf16") -> float:
    """max over elements of |got - ref| - (2e-2 + half_ulp(ref)); <= 0 passes."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) - (TOL_ABS + half_ulp(ref, dtype))))


def stat_excess(got, ref) -> float:
    """Worst margin of a statistic to its gate (<= 0 passes): relative 1e-3
    where |ref| >= 1e-3, absolute 1e-6 below; -inf (empty rows) must match."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), "rows without visible keys differ"
    keep = ~np.isneginf(ref)
    g, r = got[keep], ref[keep]
    if g.size == 0:
        return 0.0
    bound = np.where(np.abs(r) >= STAT_FLOOR, TOL_STAT * np.abs(r), TOL_STAT * STAT_FLOOR)
    return float(np.max(np.abs(g - r) - bound))


def record(case: str, tensor: str, got, ref, excess: float):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    fin = np.isfinite(ref)
    ma = max_abs(got[fin], ref[fin]) if fin.any() else 0.0
    REPORT.append((case, tensor, ma, excess, rel_l2(got[fin], ref[fin]) if fin.any() else 0.0))


def check_tensor(case: str, tensor: str, got, ref, dtype: str = "bf16", tol_l2: float | None = None):
    """Element gate (and, when given, the relative-L2 gate) on one output tensor."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), (case, tensor, "non-finite values")
    ex = elem_excess(got, ref, dtype)
    record(case, tensor, got, ref, ex)
    assert ex <= 0.0, (case, tensor, "element gate", ex, max_abs(got, ref))
    if tol_l2 is not None:
        e = rel_l2(got, ref)
        assert e <= tol_l2, (case, tensor, "relative L2", e)


def check_stat(case: str, tensor: str, got, ref):
    ex = stat_excess(got, ref)
    record(case, tensor, got, ref, ex)
    assert ex <= 0.0, (case, tensor, "statistics gate", ex)


def out_dtype(geom) -> str:
    return getattr(geom, "dtype", "bf16") or "bf16"


def format_report() -> list:
    lines = ["parity report: case | tensor | max |got-ref| | margin to gate (<= 0 passes) | rel L2"]
    for case, tensor, ma, ex, l2 in REPORT:
        lines.append(f"  {case} | {tensor} | {ma:.3e} | {ex:+.3e} | {l2:.2e}")
    return lines
