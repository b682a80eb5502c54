"""Seeded synthetic workloads for sliding-window attention.

This module only draws inputs: shapes, seeds, random tensors and the packed
dropout-keep mask.  It holds none of the attention arithmetic and is the one
module that both the CUDA path's tests and the CPU oracle's tests use.

Recipe (every workload): ``g = torch.Generator('cpu').manual_seed(seed)``;
for a TND workload the sequence lengths are drawn first
(``torch.randint(lo, hi + 1, (B,), generator=g)``); then q, k, v, dy are drawn
in that order as ``torch.randn(shape, generator=g)`` (fp32) and rounded to
bf16 (fp16 for a geometry whose dtype is "fp16"); finally, when ``keep_prob < 1``, the keep mask is drawn head by head as
``torch.rand(Sq*Skv, generator=g) < keep_prob`` in (b, n) order and packed
8 per byte, least significant bit first (element e is bit e & 7 of byte
e >> 3, 1 = keep), matching the UINT8 = 8 x 1-bit layout of the dropout mask
in the FlashAttentionVarLenScore doc (dropMaskOptional).
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict

import numpy as np
import torch

INT32_MAX = 2147483647


@dataclass
class Geometry:
    layout: str  # "BNSD" or "TND"
    B: int
    N: int
    D: int
    S_q: int = 0  # BNSD
    S_kv: int = 0
    cu_seqlens_q: list = field(default_factory=list)  # TND: cumulative ends, no leading 0
    cu_seqlens_kv: list = field(default_factory=list)
    scale: float = 1.0
    pre_tokens: int = INT32_MAX
    next_tokens: int = INT32_MAX
    sparse_mode: int = 0
    keep_prob: float = 1.0
    N_kv: int = 0  # key/value heads (grouped-query attention); 0 means N
    dropout_gen: int = 0  # 1: the keep mask is the one dropout_seed / dropout_offset stand for
    dropout_seed: int = 0
    dropout_offset: int = 0
    dtype: str = "bf16"  # element type of q, k, v, dy (and of out and the gradients): "bf16" or "fp16"

    def as_dict(self) -> dict:
        return asdict(self)

    @property
    def n_kv(self) -> int:
        return self.N_kv or self.N

    @property
    def T_q(self) -> int:
        return max(self.cu_seqlens_q) if self.cu_seqlens_q else 0

    @property
    def T_kv(self) -> int:
        return max(self.cu_seqlens_kv) if self.cu_seqlens_kv else 0

    def q_shape(self):
        return (self.B, self.N, self.S_q, self.D) if self.layout == "BNSD" else (self.T_q, self.N, self.D)

    def kv_shape(self):
        return (self.B, self.n_kv, self.S_kv, self.D) if self.layout == "BNSD" else (self.T_kv, self.n_kv, self.D)

    def stat_shape(self):
        return (self.B, self.N, self.S_q) if self.layout == "BNSD" else (self.T_q, self.N)

    def seq_lens(self):
        """(Sq_b, Skv_b) per batch; trailing zeros in a cumulative array mean 'skipped'."""
        if self.layout == "BNSD":
            return [(self.S_q, self.S_kv)] * self.B
        out, pq, pk = [], 0, 0
        for eq, ek in zip(self.cu_seqlens_q, self.cu_seqlens_kv):
            out.append((max(0, eq - pq), max(0, ek - pk)))
            pq, pk = eq, ek
        return out

    def mask_bits(self) -> int:
        return sum(self.N * a * b for a, b in self.seq_lens())


@dataclass
class Workload:
    name: str
    geom: Geometry
    seed: int
    lengths: tuple | None = None  # TND: (count, lo, hi) for the seeded length draw
    note: str = ""


def _bnsd(B, N, S, D, **kw):
    return Geometry("BNSD", B, N, D, S_q=S, S_kv=S, **kw)


# The five workloads: shapes, masks and seeds.  Seeds are 42 + k.
WORKLOADS = {
    "bnsd_1x2x256x64_nomask": Workload(
        "bnsd_1x2x256x64_nomask", _bnsd(1, 2, 256, 64, scale=1 / 8, sparse_mode=0), 43),
    "bnsd_2x16x4096x128_band2047": Workload(
        "bnsd_2x16x4096x128_band2047",
        _bnsd(2, 16, 4096, 128, scale=128 ** -0.5, sparse_mode=4, pre_tokens=2047, next_tokens=0), 44),
    "tnd_8xU512_8192_n32_d128_nomask": Workload(
        "tnd_8xU512_8192_n32_d128_nomask",
        Geometry("TND", 8, 32, 128, scale=128 ** -0.5, sparse_mode=0), 45, lengths=(8, 512, 8192)),
    "bnsd_1x32x32768x128_band4096": Workload(
        "bnsd_1x32x32768x128_band4096",
        _bnsd(1, 32, 32768, 128, scale=128 ** -0.5, sparse_mode=4, pre_tokens=4096, next_tokens=0), 46),
    "bnsd_4x16x2048x64_band256_256_drop0.9": Workload(
        "bnsd_4x16x2048x64_band256_256_drop0.9",
        _bnsd(4, 16, 2048, 64, scale=64 ** -0.5, sparse_mode=4, pre_tokens=256, next_tokens=256, keep_prob=0.9),
        47),
}
WORKLOAD_ORDER = list(WORKLOADS)
# The long sliding-window workload the throughput figure is quoted on.
HEADLINE = "bnsd_1x32x32768x128_band4096"


def pack_bits_lsb_first(keep: np.ndarray) -> np.ndarray:
    """Pack a flat bool array 8 per byte, element e -> bit (e & 7) of byte e >> 3."""
    return np.packbits(np.asarray(keep, dtype=bool).reshape(-1), bitorder="little")


@dataclass
class Inputs:
    geom: Geometry
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    dy: torch.Tensor
    drop_mask: torch.Tensor | None  # uint8, packed; None when keep_prob == 1


def draw(geom: Geometry, seed: int, lengths: tuple | None = None, with_dy: bool = True,
         mask_keep: float | None = None) -> Inputs:
    """Draw the inputs of one problem by the module recipe.

    ``lengths=(count, lo, hi)`` replaces the geometry's cumulative arrays by a
    seeded draw of ``count`` lengths in [lo, hi] (Sq = Skv per sequence).
    ``mask_keep`` forces a mask even when keep_prob == 1 (probability of 1s).
    """
    g = torch.Generator("cpu").manual_seed(int(seed))
    if lengths is not None:
        count, lo, hi = lengths
        lens = torch.randint(lo, hi + 1, (count,), generator=g).tolist()
        cu = np.cumsum(lens).tolist()
        geom = Geometry(**{**geom.as_dict(), "B": count, "cu_seqlens_q": cu, "cu_seqlens_kv": list(cu)})
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[geom.dtype]
    q = torch.randn(geom.q_shape(), generator=g).to(dt)
    k = torch.randn(geom.kv_shape(), generator=g).to(dt)
    v = torch.randn(geom.kv_shape(), generator=g).to(dt)
    dy = torch.randn(geom.q_shape(), generator=g).to(dt) if with_dy else None
    p_keep = geom.keep_prob if mask_keep is None else mask_keep
    mask = None
    if (geom.keep_prob < 1.0 and not geom.dropout_gen) or mask_keep is not None:
        chunks = []
        for (lq, lk) in geom.seq_lens():
            for _ in range(geom.N):
                if lq * lk:
                    chunks.append((torch.rand(lq * lk, generator=g) < p_keep).numpy())
        flat = np.concatenate(chunks) if chunks else np.zeros(0, dtype=bool)
        mask = torch.from_numpy(pack_bits_lsb_first(flat).copy())
    return Inputs(geom, q, k, v, dy, mask)


def draw_workload(name: str) -> Inputs:
    w = WORKLOADS[name]
    return draw(w.geom, w.seed, w.lengths)


def workload_geometry(name: str) -> Geometry:
    """The geometry draw_workload(name) uses (sequence lengths drawn from the
    workload's seed the same way), without drawing its tensors."""
    w = WORKLOADS[name]
    if w.lengths is None:
        return w.geom
    g = torch.Generator("cpu").manual_seed(int(w.seed))
    count, lo, hi = w.lengths
    cu = np.cumsum(torch.randint(lo, hi + 1, (count,), generator=g).tolist()).tolist()
    return Geometry(**{**w.geom.as_dict(), "B": count, "cu_seqlens_q": cu, "cu_seqlens_kv": list(cu)})


def _local_positions(geom: Geometry, q_side: bool) -> torch.Tensor:
    """Index of every row inside its own sequence, shaped to broadcast over
    the q-side ([B,N,S_q,1] / [T_q,1,1]) or k-side layout."""
    if geom.layout == "BNSD":
        S = geom.S_q if q_side else geom.S_kv
        return torch.arange(S, dtype=torch.float32).view(1, 1, S, 1)
    pos = []
    for lq, lk in geom.seq_lens():
        pos.append(torch.arange(lq if q_side else lk, dtype=torch.float32))
    return torch.cat(pos).view(-1, 1, 1)


def edge_probe_inputs(geom: Geometry, k_rand: torch.Tensor, dy_rand: torch.Tensor, alpha: float):
    """q, k, v, dy (bf16, D >= 8) that put each query row's probability at one
    edge of its visible window, with exact scores.

    With i, j the positions inside the sequence and s_j = 1 - 2 (j mod 2):
        q_i  = alpha * (1, 256, -(i mod 256), -256 * (i div 256), 0, ...)
        k_j  = (j mod 256, j div 256, 1, 1, r_j)
        v_j  = (s_j, 0, ...)
        dy_i = (1, 0, 0, 0, u_i)
    where r_j and u_i are the last D - 4 columns of k_rand and dy_rand.  The
    entries of q and k are integers below 2^15 (exact in bf16), so
    q_i.k_j = alpha * (j - i) exactly in fp32.  With alpha = +-1 and scale
    ln 2 the probability of key j in row i halves per key away from the
    leftmost visible key (alpha < 0) or the rightmost (alpha > 0): the
    probabilities are powers of two to within 2^-w of a w-key window, exact
    in bf16, so thousands of rows sharing one edge key (a window clipped at
    the sequence start) add no common rounding error.  dy_i.v_j = s_j alternates
    from key to key, so the row's dS at its edge key is never small, and
    out = P v stays within [-1, 1]."""
    assert geom.D >= 8 and geom.dtype == "bf16"
    i = _local_positions(geom, True)
    j = _local_positions(geom, False)
    q = torch.zeros(geom.q_shape(), dtype=torch.float32)
    qi = torch.cat([torch.ones_like(i), 256.0 * torch.ones_like(i), -torch.remainder(i, 256.0),
                    -256.0 * torch.div(i, 256.0, rounding_mode="floor")], dim=-1)
    q[..., :4] = alpha * qi
    k = k_rand.float().clone()
    k[..., 0:1] = torch.remainder(j, 256.0)
    k[..., 1:2] = torch.div(j, 256.0, rounding_mode="floor")
    k[..., 2:4] = 1.0
    v = torch.zeros(geom.kv_shape(), dtype=torch.float32)
    v[..., 0:1] = 1.0 - 2.0 * torch.remainder(j, 2.0)
    dy = dy_rand.float().clone()
    dy[..., 0] = 1.0
    dy[..., 1:4] = 0.0
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, dy))
