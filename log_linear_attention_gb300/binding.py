"""Thin ctypes binding of liblla.so (include/lla.h) for torch tensors.

Argument marshalling only: every step of the operator runs in the library's
CUDA kernels. torch supplies device memory and the current stream. The
library must exist (built by ``log_linear_attention_gb300.build``); there is
no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "liblla.so")

LLA_OK = 0
LLA_ERR_INVALID_ARG = -1
LLA_ERR_UNSUPPORTED = -2
LLA_ERR_CUDA = -3
LLA_ERR_TIMEOUT = -4
LLA_ERR_NOMEM = -5
LLA_ERR_DEVICE = -6
LLA_BF16 = 0
LLA_F32 = 1

_lock = threading.Lock()
_lib = None


class LLAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


def load() -> ctypes.CDLL:
    """Load liblla.so (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with log_linear_attention_gb300.build.build()")
            lib = ctypes.CDLL(LIB_PATH)
            vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.lla_status_string.argtypes = [i]
            lib.lla_status_string.restype = ctypes.c_char_p
            lib.lla_num_levels.argtypes = [ctypes.c_int64]
            lib.lla_num_levels.restype = i
            lib.lla_forward.argtypes = [vp, vp, vp, fp, fp, vp] + [i] * 6 + [vp, i]
            lib.lla_forward.restype = i
            lib.lla_forward_workspace_size.argtypes = [i] * 7
            lib.lla_forward_workspace_size.restype = sz
            lib.lla_forward_host.argtypes = [vp, vp, vp, fp, fp, vp] + [i] * 6 + [vp, i]
            lib.lla_forward_host.restype = i
            lib.lla_forward_ws.argtypes = [vp, vp, vp, fp, fp, vp] + [i] * 6 + [vp, i, vp, sz]
            lib.lla_forward_ws.restype = i
            lib.lla_forward_noalloc.argtypes = [vp, vp, vp, fp, fp, vp] + [i] * 6 + [vp, i]
            lib.lla_forward_noalloc.restype = i
            lib.lla_forward_profile.argtypes = [vp, vp, vp, fp, fp, vp] + [i] * 6 + [vp, i, vp, vp, i]
            lib.lla_forward_profile.restype = i
            lib.lla_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, vp, vp, vp] + [i] * 6
            lib.lla_decode_step.restype = i
            lib.lla_prefill_state.argtypes = [vp, vp, fp, fp] + [i] * 6 + [vp, i]
            lib.lla_prefill_state.restype = i
            lib.lla_device_error.argtypes = [vp]
            lib.lla_device_error.restype = i
            lib.lla_gdn_forward.argtypes = [vp, vp, vp, fp, fp, fp, vp] + [i] * 6 + [vp, i]
            lib.lla_gdn_forward.restype = i
            lib.lla_gdn_decode_step.argtypes = [vp, vp, vp, fp, fp, fp, fp, vp, vp, vp] + [i] * 6
            lib.lla_gdn_decode_step.restype = i
            lib.lla_gdn_forward_profile.argtypes = [vp, vp, vp, fp, fp, fp, vp] + [i] * 6 + [vp, i, vp, vp, i]
            lib.lla_gdn_forward_profile.restype = i
            lib.lla_debug_set_waits.argtypes = [ctypes.c_int64, i]
            lib.lla_debug_set_waits.restype = i
            lib.lla_backward.argtypes = [vp, vp, vp, fp, fp, vp, vp, vp, vp, fp, fp] + [i] * 6 + [vp, i]
            lib.lla_backward.restype = i
            lib.lla_forward_varlen.argtypes = [vp, vp, vp, fp, fp, vp, vp] + [i] * 7 + [vp, i]
            lib.lla_forward_varlen.restype = i
            lib.lla_prefill_state_varlen.argtypes = [vp, vp, fp, vp, fp] + [i] * 7 + [vp, i]
            lib.lla_prefill_state_varlen.restype = i
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().lla_status_string(int(status)).decode()


def num_levels(T: int) -> int:
    return int(load().lla_num_levels(int(T)))


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return LLA_BF16
    if t.dtype == torch.float32:
        return LLA_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _stream_handle(stream) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check(t, name, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _call(status: int, where: str):
    if status != LLA_OK:
        raise LLAError(status, where)


def forward(q, k, v, log_a, lam, chunk: int, out=None, stream=None, workspace=None):
    """Chunk-parallel prefill, lla_forward / lla_forward_ws.

    q, k [B,H,T,dk]; v [B,H,T,dv] (bf16 or fp32, same dtype); log_a [B,H,T] fp32;
    lam [B,H,T,L] fp32 with L = num_levels(T). Host (CPU) inputs go through
    lla_forward_host (pipelined copies in and out) and the result comes back in host memory.
    ``workspace``: optional uint8 CUDA tensor of at least workspace_size(...) bytes.
    """
    torch = _torch()
    if not q.is_cuda:
        return _forward_host(q, k, v, log_a, lam, chunk, out, stream)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda")):
        _check(t_, n, q.device)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if log_a.dtype != torch.float32 or lam.dtype != torch.float32:
        raise TypeError("log_a and lambda must be float32")
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or log_a.shape != (B, H, T) or lam.shape[:3] != (B, H, T):
        raise ValueError("shape mismatch between q, k, v, log_a and lambda")
    if lam.shape[3] != num_levels(T):
        raise ValueError(f"lambda needs {num_levels(T)} levels for T={T}, got {lam.shape[3]}")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.device)
    code = _dtype_code(q)
    lib = load()
    sh = _stream_handle(stream)
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(), out.data_ptr(),
            B, H, T, dk, dv, int(chunk), sh, code)
    if workspace is None:
        _call(lib.lla_forward(*args), "lla_forward")
    else:
        _check(workspace, "workspace", q.device)
        _call(lib.lla_forward_ws(*args, workspace.data_ptr(), workspace.numel() * workspace.element_size()),
              "lla_forward_ws")
    return out


def _forward_host(q, k, v, log_a, lam, chunk, out=None, stream=None):
    """lla_forward_host: every tensor in host memory (pinned for full copy bandwidth). The
    library copies head groups in, runs them and copies them out with the copies of one group
    overlapping the kernels of the next; returns the host output (pinned unless given)."""
    torch = _torch()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda")):
        if t_.is_cuda or not t_.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    if k.dtype != q.dtype or v.dtype != q.dtype or log_a.dtype != torch.float32 or lam.dtype != torch.float32:
        raise TypeError("q, k, v share one dtype; log_a and lambda are float32")
    if k.shape != q.shape or v.shape[:3] != (B, H, T) or log_a.shape != (B, H, T) or lam.shape != (B, H, T, num_levels(T)):
        raise ValueError("shape mismatch between q, k, v, log_a and lambda")
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, pin_memory=True)
    if out.is_cuda or not out.is_contiguous() or out.shape != (B, H, T, dv) or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous host tensor [B,H,T,dv] of q's dtype")
    _call(load().lla_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                                  out.data_ptr(), B, H, T, dk, dv, int(chunk), _stream_handle(stream),
                                  _dtype_code(q)), "lla_forward_host")
    return out


NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024


def forward_noalloc(q, k, v, log_a, lam, chunk: int, out, stream=None):
    """lla_forward_noalloc: the prefill with its scratch in the library's fixed device
    array (no allocation at all). ``out`` must be preallocated by the caller. Raises
    LLAError(LLA_ERR_NOMEM) when the sizes need more than NOALLOC_SCRATCH_BYTES."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda"), (out, "out")):
        _check(t_, n, q.device)
    _call(load().lla_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                                     out.data_ptr(), B, H, T, dk, dv, int(chunk), _stream_handle(stream),
                                     _dtype_code(q)), "lla_forward_noalloc")
    return out


def forward_profile(q, k, v, log_a, lam, chunk: int, out, stream=None):
    """lla_forward_profile: one synchronous forward call; returns [(kernel_name, ms), ...]
    in launch order, timed with CUDA events on the launch stream."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cap = 32
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = load().lla_forward_profile(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                                   out.data_ptr(), B, H, T, dk, dv, int(chunk), _stream_handle(stream),
                                   _dtype_code(q), ctypes.cast(ms, ctypes.c_void_p),
                                   ctypes.cast(names, ctypes.c_void_p), cap)
    if n < 0:
        raise LLAError(n, "lla_forward_profile")
    return [(names[i].decode(), float(ms[i])) for i in range(min(n, cap))]


def gdn_forward(q, k, v, log_a, beta, lam, chunk: int, out=None, stream=None):
    """Log-linear Gated DeltaNet prefill, lla_gdn_forward: as ``forward`` plus ``beta`` [B,H,T] fp32."""
    torch = _torch()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        out = torch.empty((B, H, T, dv), dtype=q.dtype, device=q.device)
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (beta, "beta"), (lam, "lambda"), (out, "out")):
        _check(t_, n, q.device)
    _call(load().lla_gdn_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), beta.data_ptr(),
                                 lam.data_ptr(), out.data_ptr(), B, H, T, dk, dv, int(chunk), _stream_handle(stream),
                                 _dtype_code(q)), "lla_gdn_forward")
    return out


def gdn_forward_profile(q, k, v, log_a, beta, lam, chunk: int, out, stream=None):
    """lla_gdn_forward_profile: one synchronous call; returns [(kernel_name, ms), ...] in launch order."""
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    cap = 32
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = load().lla_gdn_forward_profile(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), beta.data_ptr(),
                                       lam.data_ptr(), out.data_ptr(), B, H, T, dk, dv, int(chunk),
                                       _stream_handle(stream), _dtype_code(q), ctypes.cast(ms, ctypes.c_void_p),
                                       ctypes.cast(names, ctypes.c_void_p), cap)
    if n < 0:
        raise LLAError(n, "lla_gdn_forward_profile")
    return [(names[i].decode(), float(ms[i])) for i in range(min(n, cap))]


def gdn_decode_step(q, k, v, log_a, beta, lam, states, t, out=None, stream=None):
    """One log-linear Gated DeltaNet decode step, lla_gdn_decode_step (states updated in place)."""
    torch = _torch()
    B, H, dk = q.shape
    dv = v.shape[-1]
    Lmax = states.shape[2]
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (beta, "beta"), (lam, "lambda"),
                  (states, "states"), (t, "t"), (out, "out")):
        _check(t_, n, q.device)
    _call(load().lla_gdn_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), beta.data_ptr(),
                                     lam.data_ptr(), states.data_ptr(), t.data_ptr(), out.data_ptr(),
                                     _stream_handle(stream), B, H, dk, dv, Lmax, _dtype_code(q)),
          "lla_gdn_decode_step")
    return out


def debug_set_waits(limit_cycles: int, hold: bool) -> None:
    """lla_debug_set_waits: test hook of the bounded waits (see include/lla.h)."""
    _call(load().lla_debug_set_waits(int(limit_cycles), 1 if hold else 0), "lla_debug_set_waits")


def workspace_size(B: int, H: int, T: int, dk: int, dv: int, chunk: int, dtype) -> int:
    """Bytes of caller-owned workspace lla_forward_ws needs (0 for invalid sizes)."""
    torch = _torch()
    code = LLA_BF16 if dtype == torch.bfloat16 else LLA_F32
    return int(load().lla_forward_workspace_size(B, H, T, dk, dv, int(chunk), code))


def decode_step(q, k, v, log_a, lam, states, t, out=None, stream=None):
    """One recurrent decode step, lla_decode_step. ``states`` [B,H,Lmax,dk,dv] fp32 is
    updated in place; ``t`` int64 [B] on the device. Returns out [B,H,dv]."""
    torch = _torch()
    B, H, dk = q.shape
    dv = v.shape[-1]
    Lmax = states.shape[2]
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda"), (states, "states"), (t, "t")):
        _check(t_, n, q.device)
    if states.dtype != torch.float32 or states.shape != (B, H, Lmax, dk, dv):
        raise ValueError("states must be float32 [B,H,Lmax,dk,dv]")
    if t.dtype != torch.int64 or t.shape != (B,):
        raise ValueError("t must be int64 [B]")
    if lam.shape != (B, H, Lmax) or log_a.shape != (B, H) or k.shape != q.shape or v.shape[:2] != (B, H):
        raise ValueError("shape mismatch in decode inputs")
    if out is None:
        out = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.device)
    _call(load().lla_decode_step(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                                 states.data_ptr(), t.data_ptr(), out.data_ptr(), _stream_handle(stream),
                                 B, H, dk, dv, Lmax, _dtype_code(q)), "lla_decode_step")
    return out


def prefill_state(k, v, log_a, states, stream=None):
    """lla_prefill_state: write into ``states`` [B,H,Lmax,dk,dv] fp32 the Fenwick state set after
    the prompt (k [B,H,T,dk], v [B,H,T,dv], log_a [B,H,T]); the next decode position is t = T."""
    torch = _torch()
    B, H, T, dk = k.shape
    dv = v.shape[-1]
    Lmax = states.shape[2]
    for t_, n in ((k, "k"), (v, "v"), (log_a, "log_a"), (states, "states")):
        _check(t_, n, k.device)
    if states.dtype != torch.float32 or states.shape != (B, H, Lmax, dk, dv):
        raise ValueError("states must be float32 [B,H,Lmax,dk,dv]")
    _call(load().lla_prefill_state(k.data_ptr(), v.data_ptr(), log_a.data_ptr(), states.data_ptr(), B, H, T, dk, dv,
                                   Lmax, _stream_handle(stream), _dtype_code(k)), "lla_prefill_state")
    return states


def backward(q, k, v, log_a, lam, dout, chunk: int, stream=None):
    """lla_backward: gradients of sum(dout * forward(q, k, v, log_a, lam)).

    Device tensors with the shapes and dtypes of lla_forward's inputs; dout like the output.
    Returns (dq, dk, dv, dlog_a, dlambda): dq/dk/dv in q's dtype, dlog_a/dlambda fp32."""
    torch = _torch()
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    for t_, n in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda"), (dout, "dout")):
        _check(t_, n, q.device)
    if k.dtype != q.dtype or v.dtype != q.dtype or dout.dtype != q.dtype:
        raise TypeError("q, k, v and dout must share one dtype")
    if log_a.dtype != torch.float32 or lam.dtype != torch.float32:
        raise TypeError("log_a and lambda must be float32")
    if (k.shape != q.shape or v.shape[:3] != (B, H, T) or dout.shape != v.shape or log_a.shape != (B, H, T)
            or lam.shape[:3] != (B, H, T)):
        raise ValueError("shape mismatch between q, k, v, dout, log_a and lambda")
    if lam.shape[3] != num_levels(T):
        raise ValueError(f"lambda needs {num_levels(T)} levels for T={T}, got {lam.shape[3]}")
    dq = torch.empty_like(q)
    dk_ = torch.empty_like(k)
    dv_ = torch.empty_like(v)
    dla = torch.empty_like(log_a)
    dlam = torch.empty_like(lam)
    _call(load().lla_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                              dout.data_ptr(), dq.data_ptr(), dk_.data_ptr(), dv_.data_ptr(), dla.data_ptr(),
                              dlam.data_ptr(), B, H, T, dk, dv, chunk, _stream_handle(stream), _dtype_code(q)),
          "lla_backward")
    return dq, dk_, dv_, dla, dlam


def forward_varlen(q, k, v, log_a, lam, cu_seqlens, max_T: int, chunk: int, out=None, stream=None):
    """lla_forward_varlen: packed sequences. q, k [H,total,dk]; v [H,total,dv]; log_a [H,total];
    lam [H,total,num_levels(max_T)]; cu_seqlens int32 [n+1] on the device."""
    torch = _torch()
    H, total, dk = q.shape
    dv = v.shape[-1]
    n = cu_seqlens.numel() - 1
    for t_, nm in ((q, "q"), (k, "k"), (v, "v"), (log_a, "log_a"), (lam, "lambda"), (cu_seqlens, "cu_seqlens")):
        _check(t_, nm, q.device)
    if cu_seqlens.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    if k.shape != q.shape or v.shape[:2] != (H, total) or log_a.shape != (H, total) or lam.shape[:2] != (H, total):
        raise ValueError("shape mismatch between packed q, k, v, log_a and lambda")
    if lam.shape[2] != num_levels(max_T):
        raise ValueError(f"lambda needs {num_levels(max_T)} levels for max_T={max_T}")
    if out is None:
        out = torch.empty((H, total, dv), dtype=q.dtype, device=q.device)
    _check(out, "out", q.device)
    _call(load().lla_forward_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), log_a.data_ptr(), lam.data_ptr(),
                                    out.data_ptr(), cu_seqlens.data_ptr(), n, H, total, max_T, dk, dv, chunk,
                                    _stream_handle(stream), _dtype_code(q)), "lla_forward_varlen")
    return out


def prefill_state_varlen(k, v, log_a, cu_seqlens, max_T: int, states, stream=None):
    """lla_prefill_state_varlen: states [n,H,Lmax,dk,dv] fp32 after each packed sequence."""
    torch = _torch()
    H, total, dk = k.shape
    dv = v.shape[-1]
    n = cu_seqlens.numel() - 1
    Lmax = states.shape[2]
    for t_, nm in ((k, "k"), (v, "v"), (log_a, "log_a"), (cu_seqlens, "cu_seqlens"), (states, "states")):
        _check(t_, nm, k.device)
    if cu_seqlens.dtype != torch.int32 or states.dtype != torch.float32 or states.shape != (n, H, Lmax, dk, dv):
        raise ValueError("cu_seqlens must be int32 and states float32 [n,H,Lmax,dk,dv]")
    _call(load().lla_prefill_state_varlen(k.data_ptr(), v.data_ptr(), log_a.data_ptr(), cu_seqlens.data_ptr(),
                                          states.data_ptr(), n, H, total, max_T, dk, dv, Lmax,
                                          _stream_handle(stream), _dtype_code(k)), "lla_prefill_state_varlen")
    return states


def device_error(stream=None) -> int:
    """Synchronise ``stream``, then read and clear the device error word (an lla status)."""
    return int(load().lla_device_error(_stream_handle(stream)))
