"""Thin Python binding of libblkattn's C ABI (include/blkattn.h).

Argument marshalling only: torch tensors are turned into strided descriptors
(data pointer, sizes, strides) and the current torch stream is passed through.
Every step of the attention runs in the library's CUDA kernels; there is no
CPU or eager fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libblkattn.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_CUDA = -3
ERR_DEVICE_TIMEOUT = -4
ERR_NO_WORKSPACE = -5
ERR_SCRATCH_LIMIT = -6
STATIC_SCRATCH_BYTES = 16 * 1024 * 1024

BF16, F32, I32, I64 = 1, 2, 3, 4
_DTYPES = {torch.bfloat16: BF16, torch.float32: F32, torch.int32: I32, torch.int64: I64}

EXPORTED = ("blkattn_fwd", "blkattn_merge", "blkattn_status_string",
            "blkattn_check_device_error", "blkattn_debug_plan", "blkattn_debug_set_split_event",
            "blkattn_fwd_static_scratch", "blkattn_last_cuda_error", "blkattn_fwd_tree",
            "blkattn_spec_sample", "blkattn_fwd_window", "blkattn_bwd", "blkattn_bwd_window",
            "blkattn_debug_stall_next_decode")


class Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("sizes", ctypes.c_int64 * 4), ("strides", ctypes.c_int64 * 4), ("device", ctypes.c_int32)]


class States(ctypes.Structure):
    _fields_ = [("m", ctypes.c_void_p), ("l", ctypes.c_void_p), ("u", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("d_v", ctypes.c_int32), ("u_row_stride", ctypes.c_int64)]


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
                ("row_groups", ctypes.c_int32), ("chunk_keys", ctypes.c_int32),
                ("n_splits", ctypes.c_int32), ("tile_keys", ctypes.c_int32),
                ("ctas", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class BlkattnError(RuntimeError):
    def __init__(self, status: int, text: str):
        super().__init__(f"blkattn status {status}: {text}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load(path: str = LIB_PATH):
    """Load libblkattn.so (built by exact_blocked_attention_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"libblkattn.so is not built ({path}); run the package build first")
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            lib.blkattn_fwd.restype = ctypes.c_int
            lib.blkattn_fwd.argtypes = [P, P, P, P, P, P, ctypes.c_float, P, P, P]
            lib.blkattn_fwd_tree.restype = ctypes.c_int
            lib.blkattn_fwd_tree.argtypes = [P, P, P, P, P, P, P, ctypes.c_float, P, P, P]
            lib.blkattn_bwd.restype = ctypes.c_int
            lib.blkattn_bwd.argtypes = [P] * 6 + [ctypes.c_float] + [P] * 7
            lib.blkattn_bwd_window.restype = ctypes.c_int
            lib.blkattn_bwd_window.argtypes = [P] * 5 + [ctypes.c_int64, P, ctypes.c_float] + [P] * 7
            lib.blkattn_fwd_window.restype = ctypes.c_int
            lib.blkattn_fwd_window.argtypes = [P, P, P, P, P, ctypes.c_int64, P, ctypes.c_float, P, P, P]
            lib.blkattn_spec_sample.restype = ctypes.c_int
            lib.blkattn_spec_sample.argtypes = [P] * 8
            lib.blkattn_fwd_static_scratch.restype = ctypes.c_int
            lib.blkattn_fwd_static_scratch.argtypes = [P, P, P, P, P, P, ctypes.c_float, P, P, P]
            lib.blkattn_merge.restype = ctypes.c_int
            lib.blkattn_merge.argtypes = [P, P, P, P]
            lib.blkattn_status_string.restype = ctypes.c_char_p
            lib.blkattn_status_string.argtypes = [ctypes.c_int]
            lib.blkattn_check_device_error.restype = ctypes.c_int
            lib.blkattn_check_device_error.argtypes = [P]
            lib.blkattn_debug_plan.restype = ctypes.c_int
            lib.blkattn_debug_plan.argtypes = [ctypes.c_int64] * 6 + [ctypes.c_int32, ctypes.c_int32, P]
            lib.blkattn_debug_stall_next_decode.restype = None
            lib.blkattn_debug_stall_next_decode.argtypes = [ctypes.c_int32]
            lib.blkattn_debug_set_split_event.restype = None
            lib.blkattn_debug_set_split_event.argtypes = [P]
            lib.blkattn_last_cuda_error.restype = ctypes.c_char_p
            lib.blkattn_last_cuda_error.argtypes = []
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().blkattn_status_string(int(status)).decode()


def _check(status: int):
    if status == OK:
        return
    text = status_string(status)
    if status == ERR_INVALID_ARG:
        raise ValueError(f"blkattn: {text}")
    if status == ERR_CUDA:
        text += f" ({load().blkattn_last_cuda_error().decode()})"
    raise BlkattnError(status, text)


def describe(t: torch.Tensor | None) -> Tensor | None:
    """Strided descriptor of a tensor (no copy, no dtype conversion)."""
    if t is None:
        return None
    if t.dtype not in _DTYPES:
        raise ValueError(f"blkattn: unsupported dtype {t.dtype}")
    if t.dim() > 4:
        raise ValueError("blkattn: at most 4 dimensions")
    d = Tensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    d.device = t.device.index if t.is_cuda else -1  # host memory: refused by the library
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.sizes[i] = s
        d.strides[i] = st
    return d


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ref(x):
    return None if x is None else ctypes.byref(x)


def fwd(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale: float, out, lse, stream=None, tree=None,
        window: int = 0):
    """blkattn_fwd on torch CUDA tensors; out and lse are written in place.
    tree: None, or int64 [B, T_q] token-tree node masks (blkattn_fwd_tree).
    window: 0, or a sliding window of that many keys (blkattn_fwd_window)."""
    lib = load()
    if window:
        if tree is not None:
            raise ValueError("blkattn: a call takes a tree or a window, not both")
        descs = [describe(t) for t in (q, k, v, seqlens_k, q_logical_pos, mask_bias, out, lse)]
        st = lib.blkattn_fwd_window(*[_ref(x) for x in descs[:5]], ctypes.c_int64(int(window)), _ref(descs[5]),
                                    ctypes.c_float(scale), _ref(descs[6]), _ref(descs[7]),
                                    _stream_handle(stream) if q.is_cuda else None)
        _check(st)
        return out, lse
    if tree is not None:
        descs = [describe(t) for t in (q, k, v, seqlens_k, q_logical_pos, tree, mask_bias, out, lse)]
        st = lib.blkattn_fwd_tree(*[_ref(x) for x in descs[:7]], ctypes.c_float(scale),
                                  _ref(descs[7]), _ref(descs[8]), _stream_handle(stream) if q.is_cuda else None)
        _check(st)
        return out, lse
    descs = [describe(t) for t in (q, k, v, seqlens_k, q_logical_pos, mask_bias, out, lse)]
    st = lib.blkattn_fwd(_ref(descs[0]), _ref(descs[1]), _ref(descs[2]), _ref(descs[3]),
                         _ref(descs[4]), _ref(descs[5]), ctypes.c_float(scale),
                         _ref(descs[6]), _ref(descs[7]), _stream_handle(stream) if q.is_cuda else None)
    _check(st)
    return out, lse


def bwd(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale: float, out, lse, dout, dq, dk, dv, stream=None,
        window: int = 0):
    """blkattn_bwd (blkattn_bwd_window when window > 0) on torch CUDA tensors;
    dq, dk, dv are written in place."""
    lib = load()
    descs = [describe(t) for t in (q, k, v, seqlens_k, q_logical_pos, mask_bias, out, lse, dout, dq, dk, dv)]
    sh = _stream_handle(stream) if q.is_cuda else None
    if window:
        st = lib.blkattn_bwd_window(*[_ref(x) for x in descs[:5]], ctypes.c_int64(int(window)), _ref(descs[5]),
                                    ctypes.c_float(scale), *[_ref(x) for x in descs[6:]], sh)
    else:
        st = lib.blkattn_bwd(*[_ref(x) for x in descs[:6]], ctypes.c_float(scale),
                             *[_ref(x) for x in descs[6:]], sh)
    _check(st)
    return dq, dk, dv


def attention_backward(q, k, v, seqlens_k, q_logical_pos, out, lse, dout, mask_bias=None, scale=None,
                       stream=None, window: int = 0):
    """Allocate fp32 dq, dk, dv and call bwd (scale defaults to 1/sqrt(d))."""
    if scale is None:
        scale = q.shape[-1] ** -0.5
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(k.shape, dtype=torch.float32, device=k.device)
    dv = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    return bwd(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale, out, lse, dout, dq, dk, dv, stream, window=window)


def fwd_static_scratch(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale: float, out, lse,
                       stream=None):
    """blkattn_fwd_static_scratch: the same call as fwd, for callers that must
    not allocate device memory at call time; the per-split scratch is a fixed
    16 MiB array inside the library (shared by all calls on a device, so calls
    must not overlap on the GPU).  Raises BlkattnError with ERR_SCRATCH_LIMIT
    when the problem needs more scratch than that."""
    lib = load()
    descs = [describe(t) for t in (q, k, v, seqlens_k, q_logical_pos, mask_bias, out, lse)]
    st = lib.blkattn_fwd_static_scratch(_ref(descs[0]), _ref(descs[1]), _ref(descs[2]), _ref(descs[3]),
                                        _ref(descs[4]), _ref(descs[5]), ctypes.c_float(scale),
                                        _ref(descs[6]), _ref(descs[7]),
                                        _stream_handle(stream) if q.is_cuda else None)
    _check(st)
    return out, lse


def attention(q, k, v, seqlens_k, q_logical_pos, mask_bias=None, scale=None,
              out_dtype=torch.float32, stream=None, tree=None, window: int = 0):
    """Allocate out/lse with torch and run blkattn_fwd (blkattn_fwd_tree with
    a token tree)."""
    B, Hq, Tq, d = q.shape
    if scale is None:
        scale = d ** -0.5
    out = torch.empty((B, Hq, Tq, v.shape[3]), dtype=out_dtype, device=q.device)
    lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
    return fwd(q, k, v, seqlens_k, q_logical_pos, mask_bias, scale, out, lse, stream, tree=tree, window=window)


def spec_sample(p, q, draft, u_accept, u_sample, n_accepted=None, token=None, stream=None):
    """blkattn_spec_sample: one speculative verification step per sequence.
    p f32 [B,k+1,V], q f32 [B,k,V], draft int32 [B,k], u_accept f32 [B,k],
    u_sample int32 [B] (32 random bits).  Returns (n_accepted, token), int32 [B]."""
    lib = load()
    B = p.shape[0]
    if n_accepted is None:
        n_accepted = torch.empty(B, dtype=torch.int32, device=p.device)
    if token is None:
        token = torch.empty(B, dtype=torch.int32, device=p.device)
    descs = [describe(t) for t in (p, q, draft, u_accept, u_sample, n_accepted, token)]
    _check(lib.blkattn_spec_sample(*[_ref(d) for d in descs], _stream_handle(stream) if p.is_cuda else None))
    return n_accepted, token


def _states(m, l, u) -> States:
    s = States()
    s.m = m.data_ptr() if m.numel() else None
    s.l = None if l is None else (l.data_ptr() if l.numel() else None)
    s.u = u.data_ptr() if u.numel() else None
    s.rows = m.shape[0]
    s.d_v = u.shape[1]
    s.u_row_stride = u.stride(0)
    for t in (m, u) + (() if l is None else (l,)):
        if t.dtype != torch.float32:
            raise ValueError("blkattn: states are float32")
    if u.stride(1) != 1:
        raise ValueError("blkattn: state u must have unit column stride")
    return s


def merge(a, b, out, stream=None):
    """blkattn_merge on (m, l, u) triples of torch tensors (l may be None)."""
    lib = load()
    sa, sb, so = _states(*a), _states(*b), _states(*out)
    _check(lib.blkattn_merge(ctypes.byref(sa), ctypes.byref(sb), ctypes.byref(so), _stream_handle(stream)))
    return out


def check_device_error(stream=None) -> int:
    """Synchronise and read/clear the device error word (test hook)."""
    return int(load().blkattn_check_device_error(_stream_handle(stream)))


def stall_next_decode(cta: int) -> None:
    """Test hook: the next tcgen05 decode launch stops CTA ``cta`` (mod the
    CTA count) at a wait nothing completes; its bounded waits run out and
    check_device_error() then reports ERR_DEVICE_TIMEOUT."""
    load().blkattn_debug_stall_next_decode(int(cta))


def set_split_event(event) -> None:
    """Record ``event`` (a torch.cuda.Event) after the main kernel of every
    later fwd call, for timing the kernels apart; None switches it off."""
    if event is None:
        load().blkattn_debug_set_split_event(None)
        return
    event.record()  # make sure the underlying CUDA event exists
    load().blkattn_debug_set_split_event(event.cuda_event)


def debug_plan(B, Hq, Hkv, Tq, Tmax, d, dtype=torch.bfloat16, num_sms=152) -> dict:
    lib = load()
    p = Plan()
    _check(lib.blkattn_debug_plan(B, Hq, Hkv, Tq, Tmax, d, _DTYPES[dtype], num_sms, ctypes.byref(p)))
    return p.as_dict()
