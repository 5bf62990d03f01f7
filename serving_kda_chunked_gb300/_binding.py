"""ctypes binding of ``libkda.so`` over torch tensors (marshalling only).

Every step of the computation runs in the CUDA kernels behind the C ABI in
``include/kda.h``; this module only checks tensor placement, dtype and shape,
allocates outputs that the caller did not provide, and passes raw device
pointers plus the current CUDA stream.  If the compiled library is missing,
loading fails with an error -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = 1
KDA_ERR_UNSUPPORTED = 2
KDA_ERR_CUDA = 3
KDA_ERR_TIMEOUT = 4
KDA_ERR_TOO_LARGE = 5
KDA_BF16 = 0
KDA_FP32 = 1

_DTYPE_CODE = {torch.bfloat16: KDA_BF16, torch.float32: KDA_FP32}
_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    """A KDA entry point returned a non-OK status."""

    def __init__(self, fn: str, status: int):
        self.status = int(status)
        super().__init__("%s failed: %s" % (fn, status_string(status)))


def load() -> ctypes.CDLL:
    """Load ``libkda.so`` (built by ``serving_kda_chunked_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libkda.so is not built (%s); build it with "
                "`python -m serving_kda_chunked_gb300.build`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        u64 = ctypes.c_uint64
        lib.kda_prefill_chunked.argtypes = [
            vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32,
            vp, vp, vp, u64, vp]
        lib.kda_prefill_chunked.restype = ctypes.c_int
        lib.kda_gdn_prefill_chunked.argtypes = lib.kda_prefill_chunked.argtypes
        lib.kda_gdn_prefill_chunked.restype = ctypes.c_int
        lib.kda_prefill_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
        lib.kda_prefill_workspace_size.restype = u64
        lib.kda_prefill_chunked_noalloc.argtypes = [
            vp, vp, vp, vp, vp, vp, vp, i32, i64, i32, i32, i32, i32, i32, vp, vp, vp]
        lib.kda_prefill_chunked_noalloc.restype = ctypes.c_int
        lib.kda_prefill_chunked_host.argtypes = lib.kda_prefill_chunked.argtypes
        lib.kda_prefill_chunked_host.restype = ctypes.c_int
        lib.kda_prefill_host_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32, i32]
        lib.kda_prefill_host_workspace_size.restype = u64
        lib.kda_noalloc_scratch_bytes.argtypes = []
        lib.kda_noalloc_scratch_bytes.restype = u64
        lib.kda_prefill_check.argtypes = [vp, vp]
        lib.kda_prefill_check.restype = ctypes.c_int
        lib.kda_prefill_noalloc_check.argtypes = [vp]
        lib.kda_prefill_noalloc_check.restype = ctypes.c_int
        lib.kda_decode_step.argtypes = [
            vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]
        lib.kda_decode_step.restype = ctypes.c_int
        lib.kda_gdn_decode_step.argtypes = lib.kda_decode_step.argtypes
        lib.kda_gdn_decode_step.restype = ctypes.c_int
        lib.kda_decode_step_pooled.argtypes = [
            vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp]
        lib.kda_decode_step_pooled.restype = ctypes.c_int
        lib.kda_gdn_decode_step_pooled.argtypes = lib.kda_decode_step_pooled.argtypes
        lib.kda_gdn_decode_step_pooled.restype = ctypes.c_int
        lib.kda_status_string.argtypes = [i32]
        lib.kda_status_string.restype = ctypes.c_char_p
        lib.kda_abi_version.argtypes = []
        lib.kda_abi_version.restype = i32
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def abi_version() -> int:
    return int(load().kda_abi_version())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    """Raw handle of ``stream`` (default: the current stream of ``device``, or
    of the current device); a given stream must live on ``device``."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != torch.device(device):
        raise ValueError("stream is on %s, the tensors on %s" % (stream.device, device))
    return ctypes.c_void_p(int(stream.cuda_stream))


def _same_device(device, **tensors):
    """Every given tensor (None skipped) must be on ``device``: the library
    runs on one device per call and rejects memory of any other."""
    for name, t in tensors.items():
        if t is not None and t.device != device:
            raise ValueError("%s is on %s, but q is on %s: all tensors of a call must be on "
                             "one device" % (name, t.device, device))


def _check_cuda(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (the KDA kernels run on the GPU only)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def kda_prefill_workspace_size(N, T, H, dk, dv, dtype, chunk=64) -> int:
    """Workspace bytes ``kda_prefill_chunked`` needs (0: none)."""
    code = _DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().kda_prefill_workspace_size(N, T, H, dk, dv, code, chunk))


def kda_prefill_check(workspace, stream=None) -> int:
    """Synchronise the stream and return the device status of the last
    prefill that used ``workspace`` (KDA_OK or KDA_ERR_TIMEOUT)."""
    dev = None if workspace is None else workspace.device
    with torch.cuda.device(dev):
        return int(load().kda_prefill_check(_ptr(workspace), _stream(stream, dev)))


def kda_prefill_noalloc_check(stream=None, device=None) -> int:
    """Synchronise the stream and return the device status of the last
    no-allocation prefill on ``device`` (default: the current device)."""
    with torch.cuda.device(device):
        return int(load().kda_prefill_noalloc_check(_stream(stream, device)))


def _prefill(fn, gate_shape, q, k, v, g, beta, cu_seqlens, S0, chunk, o, S_T, workspace,
             stream):
    _check_cuda("q", q)
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("q must be bfloat16 or float32")
    T, H, dk = q.shape
    dv = v.shape[-1]
    _check_cuda("k", k, q.dtype, (T, H, dk))
    _check_cuda("v", v, q.dtype, (T, H, dv))
    _check_cuda("g", g, torch.float32, gate_shape(T, H, dk))
    _check_cuda("beta", beta, torch.float32, (T, H))
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = cu_seqlens.shape[0] - 1
    if S0 is not None:
        _check_cuda("S0", S0, torch.float32, (N, H, dk, dv))
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    _check_cuda("o", o, q.dtype, (T, H, dv))
    if S_T is None:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    _check_cuda("S_T", S_T, torch.float32, (N, H, dk, dv))
    need = kda_prefill_workspace_size(N, T, H, dk, dv, q.dtype, chunk)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0
    if workspace is not None:
        _check_cuda("workspace", workspace, torch.uint8)
        ws_bytes = workspace.numel()
    _same_device(q.device, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, S0=S0, o=o,
                 S_T=S_T, workspace=workspace)
    with torch.cuda.device(q.device):
        st = getattr(load(), fn)(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
            N, T, H, dk, dv, _DTYPE_CODE[q.dtype], int(chunk), _ptr(o), _ptr(S_T),
            _ptr(workspace), ws_bytes, _stream(stream, q.device))
    if st != KDA_OK:
        raise KdaError(fn, st)
    return o, S_T


def _check_host(name, t, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cpu":
        raise ValueError("%s must be a host (CPU) tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def kda_prefill_host_workspace_size(N, T, H, dk, dv, dtype, chunk=64) -> int:
    """Device workspace bytes ``kda_prefill_chunked_host`` needs."""
    code = _DTYPE_CODE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().kda_prefill_host_workspace_size(N, T, H, dk, dv, code, chunk))


def kda_prefill_chunked_host(q, k, v, g, beta, cu_seqlens, S0=None, *, chunk: int = 64,
                             o=None, S_T=None, workspace=None, device=None, stream=None):
    """``kda_prefill_chunked`` over HOST tensors (``kda_prefill_chunked_host``
    in kda.h): q, k, v, g, beta, cu_seqlens, S0 and the outputs o, S_T are CPU
    tensors (page-locked ones let the copies overlap the kernels); the call
    copies them to and from the GPU itself.  ``workspace`` is a CUDA uint8
    tensor (allocated on ``device``, default the current one, if omitted).
    Returns (o, S_T); they are complete once ``stream`` has reached this call's
    end (synchronise before reading them)."""
    _check_host("q", q)
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("q must be bfloat16 or float32")
    T, H, dk = q.shape
    dv = v.shape[-1]
    _check_host("k", k, q.dtype, (T, H, dk))
    _check_host("v", v, q.dtype, (T, H, dv))
    _check_host("g", g, torch.float32, (T, H, dk))
    _check_host("beta", beta, torch.float32, (T, H))
    _check_host("cu_seqlens", cu_seqlens, torch.int32)
    N = cu_seqlens.shape[0] - 1
    if S0 is not None:
        _check_host("S0", S0, torch.float32, (N, H, dk, dv))
    pin = q.is_pinned()
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, pin_memory=pin)
    _check_host("o", o, q.dtype, (T, H, dv))
    if S_T is None:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, pin_memory=pin)
    _check_host("S_T", S_T, torch.float32, (N, H, dk, dv))
    if workspace is None:
        need = kda_prefill_host_workspace_size(N, T, H, dk, dv, q.dtype, chunk)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _check_cuda("workspace", workspace, torch.uint8)
    with torch.cuda.device(workspace.device):
        st = load().kda_prefill_chunked_host(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
            N, T, H, dk, dv, _DTYPE_CODE[q.dtype], int(chunk), _ptr(o), _ptr(S_T),
            _ptr(workspace), workspace.numel(), _stream(stream, workspace.device))
    if st != KDA_OK:
        raise KdaError("kda_prefill_chunked_host", st)
    return o, S_T


def kda_noalloc_scratch_bytes() -> int:
    """Size of the fixed device scratch behind ``kda_prefill_chunked_noalloc``."""
    return int(load().kda_noalloc_scratch_bytes())


def kda_prefill_chunked_noalloc(q, k, v, g, beta, cu_seqlens, S0=None, *, chunk: int = 64,
                                o=None, S_T=None, stream=None):
    """``kda_prefill_chunked`` without a workspace (``kda_prefill_chunked_noalloc``
    in kda.h): scratch lives in a fixed device array inside the library; calls
    that overlap on the GPU must not share it.  Outputs as ``kda_prefill_chunked``
    (pass ``o`` / ``S_T`` to keep the call free of allocation)."""
    _check_cuda("q", q)
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("q must be bfloat16 or float32")
    T, H, dk = q.shape
    dv = v.shape[-1]
    _check_cuda("k", k, q.dtype, (T, H, dk))
    _check_cuda("v", v, q.dtype, (T, H, dv))
    _check_cuda("g", g, torch.float32, (T, H, dk))
    _check_cuda("beta", beta, torch.float32, (T, H))
    _check_cuda("cu_seqlens", cu_seqlens, torch.int32)
    N = cu_seqlens.shape[0] - 1
    if S0 is not None:
        _check_cuda("S0", S0, torch.float32, (N, H, dk, dv))
    if o is None:
        o = torch.empty((T, H, dv), dtype=q.dtype, device=q.device)
    _check_cuda("o", o, q.dtype, (T, H, dv))
    if S_T is None:
        S_T = torch.empty((N, H, dk, dv), dtype=torch.float32, device=q.device)
    _check_cuda("S_T", S_T, torch.float32, (N, H, dk, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, cu_seqlens=cu_seqlens, S0=S0, o=o,
                 S_T=S_T)
    with torch.cuda.device(q.device):
        st = load().kda_prefill_chunked_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0), _ptr(cu_seqlens),
            N, T, H, dk, dv, _DTYPE_CODE[q.dtype], int(chunk), _ptr(o), _ptr(S_T),
            _stream(stream, q.device))
    if st != KDA_OK:
        raise KdaError("kda_prefill_chunked_noalloc", st)
    return o, S_T


def kda_prefill_chunked(q, k, v, g, beta, cu_seqlens, S0=None, *, chunk: int = 64,
                        o=None, S_T=None, workspace=None, stream=None):
    """Chunked KDA prefill over a packed batch (``kda_prefill_chunked`` in kda.h).

    q, k [T, H, dk] and v [T, H, dv] in bf16 or fp32 (all the same); g
    [T, H, dk] fp32 log-gates; beta [T, H] fp32; cu_seqlens [N+1] int32 on the
    device; S0 [N, H, dk, dv] fp32 or None.  Returns (o, S_T); pass ``o`` /
    ``S_T`` to write into existing buffers (``S_T`` may be ``S0``).
    ``workspace``: a uint8 CUDA tensor of at least
    ``kda_prefill_workspace_size(...)`` bytes; allocated here when omitted.
    """
    return _prefill("kda_prefill_chunked", lambda T, H, dk: (T, H, dk), q, k, v, g, beta,
                    cu_seqlens, S0, chunk, o, S_T, workspace, stream)


def kda_gdn_prefill_chunked(q, k, v, g, beta, cu_seqlens, S0=None, *, chunk: int = 64,
                            o=None, S_T=None, workspace=None, stream=None):
    """Chunked Gated DeltaNet prefill (``kda_gdn_prefill_chunked`` in kda.h):
    as ``kda_prefill_chunked`` with one log-gate per head, g [T, H] fp32."""
    return _prefill("kda_gdn_prefill_chunked", lambda T, H, dk: (T, H), q, k, v, g, beta,
                    cu_seqlens, S0, chunk, o, S_T, workspace, stream)


def _decode(fn, gate_shape, q, k, v, g, beta, S, o, stream):
    _check_cuda("q", q)
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("q must be bfloat16 or float32")
    B, H, dk = q.shape
    dv = v.shape[-1]
    _check_cuda("k", k, q.dtype, (B, H, dk))
    _check_cuda("v", v, q.dtype, (B, H, dv))
    _check_cuda("g", g, torch.float32, gate_shape(B, H, dk))
    _check_cuda("beta", beta, torch.float32, (B, H))
    _check_cuda("S", S, torch.float32, (B, H, dk, dv))
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check_cuda("o", o, q.dtype, (B, H, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, S=S, o=o)
    with torch.cuda.device(q.device):
        st = getattr(load(), fn)(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S), B, H, dk, dv,
            _DTYPE_CODE[q.dtype], _ptr(o), _stream(stream, q.device))
    if st != KDA_OK:
        raise KdaError(fn, st)
    return o


def kda_decode_step(q, k, v, g, beta, S, *, o=None, stream=None):
    """One batched KDA decode step (``kda_decode_step`` in kda.h).

    q, k [B, H, dk], v [B, H, dv] (bf16 or fp32); g [B, H, dk] fp32; beta
    [B, H] fp32; S [B, H, dk, dv] fp32, updated in place.  Returns o.
    """
    return _decode("kda_decode_step", lambda B, H, dk: (B, H, dk), q, k, v, g, beta, S, o,
                   stream)


def kda_gdn_decode_step(q, k, v, g, beta, S, *, o=None, stream=None):
    """One batched Gated DeltaNet decode step (``kda_gdn_decode_step`` in
    kda.h): as ``kda_decode_step`` with one log-gate per head, g [B, H] fp32."""
    return _decode("kda_gdn_decode_step", lambda B, H, dk: (B, H), q, k, v, g, beta, S, o,
                   stream)


def _decode_pooled(fn, gate_shape, q, k, v, g, beta, S_pool, slots, o, stream):
    _check_cuda("q", q)
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("q must be bfloat16 or float32")
    B, H, dk = q.shape
    dv = v.shape[-1]
    _check_cuda("k", k, q.dtype, (B, H, dk))
    _check_cuda("v", v, q.dtype, (B, H, dv))
    _check_cuda("g", g, torch.float32, gate_shape(B, H, dk))
    _check_cuda("beta", beta, torch.float32, (B, H))
    _check_cuda("S_pool", S_pool, torch.float32)
    if S_pool.dim() != 4 or tuple(S_pool.shape[1:]) != (H, dk, dv):
        raise ValueError("S_pool must have shape [P, %d, %d, %d]" % (H, dk, dv))
    _check_cuda("slots", slots, torch.int32, (B,))
    if o is None:
        o = torch.empty((B, H, dv), dtype=q.dtype, device=q.device)
    _check_cuda("o", o, q.dtype, (B, H, dv))
    _same_device(q.device, k=k, v=v, g=g, beta=beta, S_pool=S_pool, slots=slots, o=o)
    with torch.cuda.device(q.device):
        st = getattr(load(), fn)(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S_pool), _ptr(slots),
            S_pool.shape[0], B, H, dk, dv, _DTYPE_CODE[q.dtype], _ptr(o),
            _stream(stream, q.device))
    if st != KDA_OK:
        raise KdaError(fn, st)
    return o


def kda_decode_step_pooled(q, k, v, g, beta, S_pool, slots, *, o=None, stream=None):
    """Batched decode over a pool of states (``kda_decode_step_pooled`` in kda.h).

    S_pool [P, H, dk, dv] fp32; slots [B] int32 on the device (a value outside
    [0, P) skips that sequence).  The named slots are updated in place.
    Returns o [B, H, dv].
    """
    return _decode_pooled("kda_decode_step_pooled", lambda B, H, dk: (B, H, dk), q, k, v, g,
                          beta, S_pool, slots, o, stream)


def kda_gdn_decode_step_pooled(q, k, v, g, beta, S_pool, slots, *, o=None, stream=None):
    """Gated DeltaNet decode over a pool of states (``kda_gdn_decode_step_pooled``
    in kda.h): as ``kda_decode_step_pooled`` with g [B, H] fp32."""
    return _decode_pooled("kda_gdn_decode_step_pooled", lambda B, H, dk: (B, H), q, k, v, g,
                          beta, S_pool, slots, o, stream)
