"""Thin Python binding of libswa's C ABI (include/swa.h).

Argument marshalling only: every step of the attention computation runs in the
CUDA kernels of libswa.so.  PyTorch supplies device memory and streams.  If the
compiled library is missing, every call raises -- there is no fallback path.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libswa.so")
CHECKED_LIB_PATH = os.path.join(_PKG, "libswa_checked.so")

SWA_OK = 0
SWA_ERR_PARAM_NULLPTR = 161001
SWA_ERR_PARAM_INVALID = 161002
SWA_ERR_UNSUPPORTED = 161100
SWA_ERR_WORKSPACE = 161101
SWA_ERR_CUDA = 161102
SWA_ERR_TIMEOUT = 161103
SWA_ERR_BOUNDS = 161104
LAYOUTS = {"BNSD": 0, "TND": 1}
DTYPES = {"bf16": 0, "fp16": 1, "fp32": 2}


class SwaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"libswa status {status}: {message}")
        self.status = status


class SwaParams(ctypes.Structure):
    """Mirror of swa_params_t."""

    _fields_ = [
        ("layout", ctypes.c_int32),
        ("B", ctypes.c_int64),
        ("N", ctypes.c_int64),
        ("D", ctypes.c_int64),
        ("S_q", ctypes.c_int64),
        ("S_kv", ctypes.c_int64),
        ("T_q", ctypes.c_int64),
        ("T_kv", ctypes.c_int64),
        ("cu_seqlens_q", ctypes.POINTER(ctypes.c_int64)),
        ("cu_seqlens_kv", ctypes.POINTER(ctypes.c_int64)),
        ("scale", ctypes.c_double),
        ("pre_tokens", ctypes.c_int64),
        ("next_tokens", ctypes.c_int64),
        ("sparse_mode", ctypes.c_int32),
        ("keep_prob", ctypes.c_double),
        ("N_kv", ctypes.c_int64),
        ("dropout_gen", ctypes.c_int32),
        ("dropout_seed", ctypes.c_uint64),
        ("dropout_offset", ctypes.c_uint64),
        ("dtype", ctypes.c_int32),
    ]


_lib = None
_checked_lib = None
_lock = threading.Lock()
_local = threading.local()  # .lib: the library this thread's calls go to, when set by using()


def lib() -> ctypes.CDLL:
    """The library this thread's calls go to: libswa.so (built in-tree by
    ``build.build()``), unless ``using()`` chose another; raise if it is absent."""
    override = getattr(_local, "lib", None)
    if override is not None:
        return override
    global _lib
    with _lock:
        if _lib is None:
            _lib = _open(LIB_PATH, "attention_swa_forward_gb300.build.build()")
    return _lib


def checked_lib() -> ctypes.CDLL:
    """The bounds-checked build, libswa_checked.so (``build.build(checked=True)``):
    the same kernels with every global load and store tested against its
    tensor's extent; an access outside it is skipped and reported as
    SWA_ERR_BOUNDS by swa_workspace_status."""
    global _checked_lib
    with _lock:
        if _checked_lib is None:
            _checked_lib = _open(CHECKED_LIB_PATH, "attention_swa_forward_gb300.build.build(checked=True)")
    return _checked_lib


@contextlib.contextmanager
def using(library: ctypes.CDLL):
    """Route this thread's calls of this module to `library` (e.g. checked_lib())."""
    before = getattr(_local, "lib", None)
    _local.lib = library
    try:
        yield library
    finally:
        _local.lib = before


def _open(path: str, how: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with {how}")
    L = ctypes.CDLL(path)
    P = ctypes.POINTER(SwaParams)
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    st = ctypes.c_int
    L.swa_params_default.argtypes = [P]
    L.swa_params_default.restype = None
    L.swa_forward_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    L.swa_forward_workspace_size.restype = st
    L.swa_backward_workspace_size.argtypes = [P, ctypes.POINTER(sz)]
    L.swa_backward_workspace_size.restype = st
    L.swa_forward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.swa_forward.restype = st
    L.swa_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.swa_backward.restype = st
    L.swa_backward_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.swa_backward_noalloc.restype = st
    L.swa_workspace_status.argtypes = [vp, vp]
    L.swa_workspace_status.restype = st
    L.swa_dropout_mask.argtypes = [P, vp, sz, vp]
    L.swa_dropout_mask.restype = st
    ci = ctypes.c_int
    L.swa_step_host_buffer_size.argtypes = [P, ci, ctypes.POINTER(sz)]
    L.swa_step_host_buffer_size.restype = st
    L.swa_step_host.argtypes = [P, ci, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.swa_step_host.restype = st
    L.swa_step_host_status.argtypes = [P, ci, vp, vp]
    L.swa_step_host_status.restype = st
    L.swa_set_timing_events.argtypes = [vp]
    L.swa_set_timing_events.restype = None
    L.swa_debug_schedule.argtypes = [P, ctypes.c_int32, vp, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
    L.swa_debug_schedule.restype = st
    L.swa_debug_stall.argtypes = [ctypes.c_int32]
    L.swa_debug_stall.restype = None
    L.swa_debug_forward_pairs.argtypes = [ctypes.c_int32]
    L.swa_debug_forward_pairs.restype = None
    L.swa_debug_extent_slack.argtypes = [ctypes.c_int64]
    L.swa_debug_extent_slack.restype = None
    L.swa_last_error.argtypes = []
    L.swa_last_error.restype = ctypes.c_char_p
    return L


def exported_symbols():
    return ["swa_params_default", "swa_forward_workspace_size", "swa_forward", "swa_backward_workspace_size",
            "swa_backward", "swa_backward_noalloc", "swa_workspace_status", "swa_set_timing_events",
            "swa_last_error", "swa_dropout_mask", "swa_step_host_buffer_size", "swa_step_host",
            "swa_step_host_status", "swa_debug_schedule", "swa_debug_stall", "swa_debug_forward_pairs",
            "swa_debug_extent_slack"]


def _check(status: int):
    if status != SWA_OK:
        raise SwaError(status, lib().swa_last_error().decode())


class Params:
    """swa_params_t built from a geometry object (fields as in ``workloads.Geometry``)."""

    def __init__(self, geom):
        self.geom = geom
        self.c = SwaParams()
        lib().swa_params_default(ctypes.byref(self.c))
        c = self.c
        c.layout = LAYOUTS[geom.layout]
        c.B, c.N, c.D = geom.B, geom.N, geom.D
        self._cu_q = self._cu_kv = None
        if geom.layout == "BNSD":
            c.S_q, c.S_kv = geom.S_q, geom.S_kv
        else:
            self._cu_q = (ctypes.c_int64 * len(geom.cu_seqlens_q))(*[int(x) for x in geom.cu_seqlens_q])
            self._cu_kv = (ctypes.c_int64 * len(geom.cu_seqlens_kv))(*[int(x) for x in geom.cu_seqlens_kv])
            c.cu_seqlens_q = ctypes.cast(self._cu_q, ctypes.POINTER(ctypes.c_int64))
            c.cu_seqlens_kv = ctypes.cast(self._cu_kv, ctypes.POINTER(ctypes.c_int64))
            c.T_q = max(int(x) for x in geom.cu_seqlens_q)
            c.T_kv = max(int(x) for x in geom.cu_seqlens_kv)
        c.scale = float(geom.scale)
        c.pre_tokens = int(geom.pre_tokens)
        c.next_tokens = int(geom.next_tokens)
        c.sparse_mode = int(geom.sparse_mode)
        c.keep_prob = float(geom.keep_prob)
        c.N_kv = int(getattr(geom, "N_kv", 0) or 0)
        c.dropout_gen = int(getattr(geom, "dropout_gen", 0) or 0)
        c.dropout_seed = int(getattr(geom, "dropout_seed", 0) or 0) & (2**64 - 1)
        c.dropout_offset = int(getattr(geom, "dropout_offset", 0) or 0) & (2**64 - 1)
        c.dtype = DTYPES[getattr(geom, "dtype", "bf16") or "bf16"]

    def ref(self):
        return ctypes.byref(self.c)


# ------------------------------------------------------------ raw C calls --
def swa_forward_workspace_size(params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().swa_forward_workspace_size(params.ref(), ctypes.byref(n)))
    return n.value


def swa_backward_workspace_size(params: Params) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().swa_backward_workspace_size(params.ref(), ctypes.byref(n)))
    return n.value


def swa_forward(params: Params, q, k, v, drop_mask, out, softmax_max, softmax_sum, workspace, workspace_bytes,
                stream) -> int:
    """Raw call with integer device pointers; returns the status code."""
    return lib().swa_forward(params.ref(), q, k, v, drop_mask, out, softmax_max, softmax_sum, workspace,
                             workspace_bytes, stream)


def swa_backward(params: Params, q, k, v, dy, out, softmax_max, softmax_sum, drop_mask, dq, dk, dv, workspace,
                 workspace_bytes, stream) -> int:
    return lib().swa_backward(params.ref(), q, k, v, dy, out, softmax_max, softmax_sum, drop_mask, dq, dk, dv,
                              workspace, workspace_bytes, stream)


def swa_backward_noalloc(params: Params, q, k, v, dy, out, softmax_max, softmax_sum, drop_mask, dq, dk, dv,
                         stream) -> int:
    """Raw call of the no-allocation backward (scratch compiled into the library)."""
    return lib().swa_backward_noalloc(params.ref(), q, k, v, dy, out, softmax_max, softmax_sum, drop_mask, dq, dk,
                                      dv, stream)


def swa_workspace_status(workspace, stream) -> int:
    return lib().swa_workspace_status(workspace, stream)


def swa_dropout_mask(params: "Params", mask, mask_bytes: int, stream) -> int:
    """Raw call: write the keep mask params' dropout seed / offset stand for."""
    return lib().swa_dropout_mask(params.ref(), mask, mask_bytes, stream)


def swa_step_host_buffer_size(params: "Params", chunks: int) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().swa_step_host_buffer_size(params.ref(), int(chunks), ctypes.byref(n)))
    return n.value


def swa_step_host(params: "Params", chunks, q, k, v, dy, out, softmax_max, softmax_sum, dq, dk, dv, device_buffer,
                  device_bytes, stream) -> int:
    """Raw call: host pointers for the tensors, a device pointer for the buffer."""
    return lib().swa_step_host(params.ref(), int(chunks), q, k, v, dy, out, softmax_max, softmax_sum, dq, dk, dv,
                               device_buffer, device_bytes, stream)


_timing_handles = None


def swa_set_timing_events(events=None):
    """Eight raw cudaEvent_t handles (ints): forward, dK/dV, dQ and preprocess
    start/stop pairs; None stops recording."""
    global _timing_handles
    if events is None:
        _timing_handles = None
        lib().swa_set_timing_events(None)
        return
    _timing_handles = (ctypes.c_void_p * 8)(*events)
    lib().swa_set_timing_events(_timing_handles)


def swa_last_error() -> str:
    return lib().swa_last_error().decode()


def swa_debug_schedule(params: "Params", pass_: int):
    """The scheduler's work items of one pass as an int32 array [items, 6]:
    launch, batch, head, tile, first partner tile, partner tile count."""
    import numpy as np

    count = ctypes.c_int64(0)
    _check(lib().swa_debug_schedule(params.ref(), int(pass_), None, 0, ctypes.byref(count)))
    out = np.zeros((max(count.value, 1), 6), dtype=np.int32)
    _check(lib().swa_debug_schedule(params.ref(), int(pass_), out.ctypes.data_as(ctypes.c_void_p), count.value,
                                    ctypes.byref(count)))
    return out[:count.value]


def swa_debug_stall(kernels: int):
    """Test hook: kernels (bit 0 forward, 1 key-major, 2 query-major) whose
    compute warps first wait on a barrier nothing completes; 0 turns it off."""
    lib().swa_debug_stall(int(kernels))


def swa_debug_forward_pairs(mode: int):
    """Test hook: forward kernel choice at D <= 64 (0 by size, 1 always one
    CTA per pair of query tiles, 2 never)."""
    lib().swa_debug_forward_pairs(int(mode))


def swa_debug_extent_slack(elems: int):
    """Test hook: elements taken off every extent the bounds-checked build
    tests the kernels' accesses against (the release build ignores it); 0
    turns it off."""
    lib().swa_debug_extent_slack(int(elems))


# ------------------------------------------------------- torch convenience --
def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def forward(geom, q, k, v, drop_mask=None, out=None, softmax_max=None, softmax_sum=None, workspace=None,
            stream=None):
    """Enqueue swa_forward on device tensors; returns (out, softmax_max, softmax_sum)."""
    p = Params(geom)
    dev = q.device
    out = torch.empty_like(q) if out is None else out
    stat_shape = tuple(geom.stat_shape()) if hasattr(geom, "stat_shape") else None
    if softmax_max is None:
        softmax_max = torch.empty(stat_shape, dtype=torch.float32, device=dev)
    if softmax_sum is None:
        softmax_sum = torch.empty(stat_shape, dtype=torch.float32, device=dev)
    need = swa_forward_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(swa_forward(p, _ptr(q), _ptr(k), _ptr(v), _ptr(drop_mask), _ptr(out), _ptr(softmax_max),
                       _ptr(softmax_sum), _ptr(workspace), workspace.numel(), _stream_handle(stream)))
    return out, softmax_max, softmax_sum


def backward(geom, q, k, v, dy, out, softmax_max, softmax_sum, drop_mask=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Enqueue swa_backward on device tensors; returns (dq, dk, dv)."""
    p = Params(geom)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = swa_backward_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(swa_backward(p, _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(out), _ptr(softmax_max), _ptr(softmax_sum),
                        _ptr(drop_mask), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
                        _stream_handle(stream)))
    return dq, dk, dv


def dropout_mask(geom, device="cuda:0", stream=None):
    """The packed keep mask (uint8 device tensor, drop_mask layout, padded to
    a 16-byte multiple) that geom's dropout_seed / dropout_offset stand for."""
    nbytes = (geom.mask_bits() + 127) // 128 * 16
    mask = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    _check(swa_dropout_mask(Params(geom), _ptr(mask), mask.numel(), _stream_handle(stream)))
    return mask


def step_host(geom, q, k, v, dy, out, softmax_max, softmax_sum, dq, dk, dv, chunks=1, device_buffer=None,
              stream=None, device="cuda:0"):
    """Enqueue swa_step_host on host tensors (page-locked for overlap): forward
    and backward with the copies overlapped with the computation.  Results
    land in the given host tensors when the stream completes.  Returns the
    device buffer (reuse it for the next call)."""
    p = Params(geom)
    need = swa_step_host_buffer_size(p, chunks)
    if device_buffer is None:
        device_buffer = torch.empty(need, dtype=torch.uint8, device=device)
    _check(swa_step_host(p, chunks, _ptr(q), _ptr(k), _ptr(v), _ptr(dy), _ptr(out), _ptr(softmax_max),
                         _ptr(softmax_sum), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(device_buffer), device_buffer.numel(),
                         _stream_handle(stream)))
    return device_buffer


def check_step_host(geom, chunks, device_buffer, stream=None):
    """Wait for the stream and raise if a kernel of a swa_step_host call gave up a bounded wait."""
    _check(lib().swa_step_host_status(Params(geom).ref(), int(chunks), _ptr(device_buffer), _stream_handle(stream)))


def check_workspace(workspace, stream=None):
    """Wait for the stream and raise if a kernel gave up a bounded wait."""
    _check(swa_workspace_status(_ptr(workspace), _stream_handle(stream)))
