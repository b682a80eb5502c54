"""Python face of the fp64 CPU oracle (``swa_ref.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference arm are the only callers.  The oracle shares no code
with the CUDA path and never imports it.

Inputs are bf16 tensors (torch, CPU) or float arrays; they are converted to
float64 (exactly, for bf16 values) before the C code sees them.  Outputs are
float64 numpy arrays.  Layouts follow the attention API
of the FlashAttentionVarLenScore doc (parameter list): BNSD ``[B,N,S,D]`` or
TND ``[T,N,D]``; statistics ``[B,N,S]`` / ``[T,N]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swa_ref.c")
_LIB_PATH = os.path.join(_HERE, "libswa_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``swa_ref.c`` into ``libswa_oracle.so`` (gcc, OpenMP, -O2, no fast-math)."""
    stale = not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("layout", ctypes.c_int32),
        ("sparse_mode", ctypes.c_int32),
        ("B", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("D", ctypes.c_int64),
        ("S_q", ctypes.c_int64),
        ("S_kv", ctypes.c_int64),
        ("T_q", ctypes.c_int64),
        ("T_kv", ctypes.c_int64),
        ("cu_q", ctypes.POINTER(ctypes.c_int64)),
        ("cu_kv", ctypes.POINTER(ctypes.c_int64)),
        ("scale", ctypes.c_double),
        ("pre_tokens", ctypes.c_int64),
        ("next_tokens", ctypes.c_int64),
        ("keep_prob", ctypes.c_double),
        ("N_kv", ctypes.c_int64),
    ]


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Params)
            vp = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.orc_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_forward_rows.argtypes = [P, vp, vp, vp, vp, i64, vp, vp, vp, vp]
            lib.orc_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_backward_dq_rows.argtypes = [P, vp, vp, vp, vp, vp, i64, vp, vp]
            lib.orc_backward_dkv_cols.argtypes = [P, vp, vp, vp, vp, vp, i64, vp, vp, vp]
            lib.orc_key_ranges.argtypes = [P, i64, vp, vp, vp]
            lib.orc_rounding_budget.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            lib.orc_rounding_error.argtypes = [P, vp, vp, vp, vp, vp, ctypes.c_double, vp, vp, vp, vp]
            lib.orc_philox4x32_10.argtypes = [vp, vp, vp]
            lib.orc_philox4x32_10.restype = None
            lib.orc_generate_keep_mask.argtypes = [P, ctypes.c_uint64, ctypes.c_uint64, vp]
            _lib = lib
    return _lib


@dataclass
class Problem:
    """Geometry and attributes of one attention call (the oracle's view)."""

    layout: str  # "BNSD" or "TND"
    B: int
    N: int
    D: int
    S_q: int = 0
    S_kv: int = 0
    cu_seqlens_q: list = field(default_factory=list)  # TND: cumulative ends, no leading 0
    cu_seqlens_kv: list = field(default_factory=list)
    scale: float = 1.0
    pre_tokens: int = 2147483647
    next_tokens: int = 2147483647
    sparse_mode: int = 0
    keep_prob: float = 1.0
    N_kv: int = 0  # key/value heads (GQA / MQA); 0 means N
    # A seed / offset standing for the dropout mask: the oracle does not use
    # them directly; generate_keep_mask turns them into the mask it takes.
    dropout_gen: int = 0
    dropout_seed: int = 0
    dropout_offset: int = 0
    dtype: str = "bf16"  # the inputs' element type; the oracle reads their exact values in fp64

    @property
    def n_kv(self) -> int:
        return self.N_kv or self.N

    @property
    def T_q(self) -> int:
        return max(self.cu_seqlens_q) if self.cu_seqlens_q else 0

    @property
    def T_kv(self) -> int:
        return max(self.cu_seqlens_kv) if self.cu_seqlens_kv else 0

    def q_rows(self) -> int:
        return self.B * self.S_q if self.layout == "BNSD" else self.T_q

    def kv_rows(self) -> int:
        return self.B * self.S_kv if self.layout == "BNSD" else self.T_kv


def _as_f64(x) -> np.ndarray:
    """bf16 torch tensor (or any float array) -> contiguous float64 numpy (exact for bf16)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    return np.ascontiguousarray(x.detach().cpu().contiguous().double().numpy())


def _as_u8(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.uint8)
    return np.ascontiguousarray(x.detach().cpu().contiguous().numpy().astype(np.uint8, copy=False))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class _Call:
    """Holds the ctypes params struct and keeps its arrays alive."""

    def __init__(self, pr: Problem):
        self.cu_q = np.ascontiguousarray(np.array(pr.cu_seqlens_q or [0], dtype=np.int64))
        self.cu_kv = np.ascontiguousarray(np.array(pr.cu_seqlens_kv or [0], dtype=np.int64))
        self.p = _Params(
            0 if pr.layout == "BNSD" else 1,
            pr.sparse_mode,
            pr.B,
            pr.N,
            pr.D,
            pr.S_q,
            pr.S_kv,
            pr.T_q,
            pr.T_kv,
            self.cu_q.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            self.cu_kv.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
            pr.scale,
            pr.pre_tokens,
            pr.next_tokens,
            pr.keep_prob,
            pr.n_kv,
        )
        if pr.n_kv < 1 or pr.N % pr.n_kv:
            raise ValueError(f"N={pr.N} is not a multiple of N_kv={pr.n_kv}")

    def ref(self):
        return ctypes.byref(self.p)


def _stat_shape(pr: Problem):
    return (pr.B, pr.N, pr.S_q) if pr.layout == "BNSD" else (pr.T_q, pr.N)


def _q_shape(pr: Problem):
    return (pr.B, pr.N, pr.S_q, pr.D) if pr.layout == "BNSD" else (pr.T_q, pr.N, pr.D)


def _kv_shape(pr: Problem):
    return (pr.B, pr.n_kv, pr.S_kv, pr.D) if pr.layout == "BNSD" else (pr.T_kv, pr.n_kv, pr.D)


def forward(pr: Problem, q, k, v, drop_mask=None):
    """Full forward.  Returns (out, softmax_max, softmax_sum) as float64."""
    lib = _load()
    c = _Call(pr)
    q, k, v, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_u8(drop_mask)
    out = np.zeros(_q_shape(pr), dtype=np.float64)
    smax = np.full(_stat_shape(pr), -np.inf, dtype=np.float64)
    ssum = np.zeros(_stat_shape(pr), dtype=np.float64)
    lib.orc_forward(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(m), _ptr(out), _ptr(smax), _ptr(ssum))
    return out, smax, ssum


def forward_rows(pr: Problem, q, k, v, drop_mask, rows):
    """Forward for selected query rows (flat statistics ids).  Returns
    (out[n, D], softmax_max[n], softmax_sum[n])."""
    lib = _load()
    c = _Call(pr)
    q, k, v, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_u8(drop_mask)
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.zeros((len(sel), pr.D), dtype=np.float64)
    smax = np.zeros(len(sel), dtype=np.float64)
    ssum = np.zeros(len(sel), dtype=np.float64)
    lib.orc_forward_rows(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(m), len(sel), _ptr(sel), _ptr(out), _ptr(smax),
                         _ptr(ssum))
    return out, smax, ssum


def backward(pr: Problem, q, k, v, dy, drop_mask=None, given_out=None, given_max=None, given_sum=None):
    """Full backward.  Exact mode (the oracle's own forward) unless the
    forward results are given.  Returns (dq, dk, dv) as float64."""
    lib = _load()
    c = _Call(pr)
    q, k, v, dy, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy), _as_u8(drop_mask)
    go, gm, gs = _as_f64(given_out), _as_f64(given_max), _as_f64(given_sum)
    dq = np.zeros(_q_shape(pr), dtype=np.float64)
    dk = np.zeros(_kv_shape(pr), dtype=np.float64)
    dv = np.zeros(_kv_shape(pr), dtype=np.float64)
    lib.orc_backward(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(m), _ptr(go), _ptr(gm), _ptr(gs), _ptr(dq),
                     _ptr(dk), _ptr(dv))
    return dq, dk, dv


def backward_dq_rows(pr: Problem, q, k, v, dy, drop_mask, rows):
    """dQ for selected query rows (flat statistics ids), exact mode."""
    lib = _load()
    c = _Call(pr)
    q, k, v, dy, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy), _as_u8(drop_mask)
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    dq = np.zeros((len(sel), pr.D), dtype=np.float64)
    lib.orc_backward_dq_rows(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(m), len(sel), _ptr(sel), _ptr(dq))
    return dq


def backward_dkv_cols(pr: Problem, q, k, v, dy, drop_mask, cols):
    """dK and dV for selected key rows (flat ids (b*N_kv+h)*S_kv+j or t*N_kv+h)."""
    lib = _load()
    c = _Call(pr)
    q, k, v, dy, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy), _as_u8(drop_mask)
    sel = np.ascontiguousarray(np.asarray(cols, dtype=np.int64))
    dk = np.zeros((len(sel), pr.D), dtype=np.float64)
    dv = np.zeros((len(sel), pr.D), dtype=np.float64)
    lib.orc_backward_dkv_cols(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(m), len(sel), _ptr(sel), _ptr(dk),
                              _ptr(dv))
    return dk, dv


def rounding_budget(pr: Problem, q, k, v, dy, drop_mask=None):
    """Test support: per element, the sums of absolute values that bound the
    drift of out, dQ, dK and dV when the products' operands P~ (forward,
    dV) and dS (dQ, dK) are rounded to a float of unit roundoff u: the error
    is at most u times the budget, to first order.  Returns (out_b, dq_b,
    dk_b, dv_b) as float64 in the layouts of out / q and k / v."""
    lib = _load()
    c = _Call(pr)
    q, k, v, dy, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy), _as_u8(drop_mask)
    out_b = np.zeros(_q_shape(pr), dtype=np.float64)
    dq_b = np.zeros(_q_shape(pr), dtype=np.float64)
    dk_b = np.zeros(_kv_shape(pr), dtype=np.float64)
    dv_b = np.zeros(_kv_shape(pr), dtype=np.float64)
    lib.orc_rounding_budget(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(m), _ptr(out_b), _ptr(dq_b),
                            _ptr(dk_b), _ptr(dv_b))
    return out_b, dq_b, dk_b, dv_b


def rounding_error(pr: Problem, q, k, v, dy, drop_mask=None, u: float = 2.0 ** -8):
    """Test support: per element, first-order error bounds of an evaluation
    that rounds P~ (forward and dV), dS (dQ and dK) and the stored output O
    to a float of unit roundoff ``u`` and computes everything else exactly:
    u times the rounding budgets, plus for dQ and dK the effect of the error
    of D_i = dY_i . O_i formed from that O.  Returns (out_e, dq_e, dk_e,
    dv_e) as float64."""
    lib = _load()
    c = _Call(pr)
    q, k, v, dy, m = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(dy), _as_u8(drop_mask)
    out_e = np.zeros(_q_shape(pr), dtype=np.float64)
    dq_e = np.zeros(_q_shape(pr), dtype=np.float64)
    dk_e = np.zeros(_kv_shape(pr), dtype=np.float64)
    dv_e = np.zeros(_kv_shape(pr), dtype=np.float64)
    lib.orc_rounding_error(c.ref(), _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(m), float(u), _ptr(out_e), _ptr(dq_e),
                           _ptr(dk_e), _ptr(dv_e))
    return out_e, dq_e, dk_e, dv_e


def key_ranges(pr: Problem, rows):
    """Visible key range [lo, hi] of each selected query row (lo > hi: empty)."""
    lib = _load()
    c = _Call(pr)
    sel = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    lo = np.zeros(len(sel), dtype=np.int64)
    hi = np.zeros(len(sel), dtype=np.int64)
    lib.orc_key_ranges(c.ref(), len(sel), _ptr(sel), _ptr(lo), _ptr(hi))
    return lo, hi


def philox4x32_10(counter, key):
    """Philox4x32-10 of a 4-word counter under a 2-word key -> 4 uint32 words."""
    lib = _load()
    c = np.ascontiguousarray(np.asarray(counter, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    out = np.zeros(4, dtype=np.uint32)
    lib.orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def generate_keep_mask(pr: Problem, seed: int, offset: int) -> np.ndarray:
    """The packed keep mask (uint8, drop_mask order) a dropout seed / offset pair stands for."""
    lib = _load()
    c = _Call(pr)
    nbits = 0
    if pr.layout == "BNSD":
        nbits = pr.B * pr.N * pr.S_q * pr.S_kv
    else:
        pq = pk = 0
        for eq, ek in zip(pr.cu_seqlens_q, pr.cu_seqlens_kv):
            nbits += pr.N * max(0, eq - pq) * max(0, ek - pk)
            pq, pk = eq, ek
    mask = np.zeros((nbits + 7) // 8, dtype=np.uint8)
    lib.orc_generate_keep_mask(c.ref(), int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(mask))
    return mask


def flops(pr: Problem) -> float:
    """Algorithmic fwd+bwd FLOPs: 14*D per visible (i, j) pair over all heads."""
    return 14.0 * pr.D * visible_pairs(pr)


def visible_pairs(pr: Problem) -> int:
    """Number of visible (i, j) pairs over all heads, by the BAND inequality."""
    total = 0
    if pr.layout == "BNSD":
        spans = [(pr.S_q, pr.S_kv)] * pr.B
    else:
        spans = []
        pq = pk = 0
        for eq, ek in zip(pr.cu_seqlens_q, pr.cu_seqlens_kv):
            spans.append((max(0, eq - pq), max(0, ek - pk)))
            pq, pk = eq, ek
    for lq, lk in spans:
        if lq == 0 or lk == 0:
            continue
        i = np.arange(lq, dtype=np.int64)
        if pr.sparse_mode == 4:
            lo = np.maximum(0, i - pr.pre_tokens)
            hi = np.minimum(lk - 1, i + pr.next_tokens)
        else:
            lo = np.zeros_like(i)
            hi = np.full_like(i, lk - 1)
        total += int(np.maximum(0, hi - lo + 1).sum())
    return total * pr.N
