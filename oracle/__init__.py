"""fp64 CPU oracle for Kimi Delta Attention (KDA) -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and it
shares no code with the CUDA library.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, POSIX threads over
independent (sequence, head, state-column block) units).  This module only
compiles it with the host C compiler and marshals numpy arrays.

Every function here follows the token recurrence of the lineage essay
"GPT-2부터 Kimi K3까지" (sections "DeltaNet", "Gated DeltaNet" and "KDA"):
decay the state by the per-channel gate, read v_old = k^T S, write
beta (v - v_old) along k, and read out o = S^T q.  Its pins (closed forms,
brute-force transition products, invariants) are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle (gcc, -O2, no -march) into ``out``; by default
    ``liboracle.so`` next to the source."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class OracleLib:
    """ctypes view of one compiled oracle library (the default one, or a
    deliberately mutated copy built by the mutation tests)."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        ip = ctypes.POINTER(ctypes.c_int64)
        lib.kda_oracle_prefill.argtypes = [
            dp, dp, dp, dp, dp, dp, ip, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, dp, dp, ctypes.c_int]
        lib.kda_oracle_prefill.restype = ctypes.c_int
        lib.kda_oracle_decode_step.argtypes = [
            dp, dp, dp, dp, dp, dp, ctypes.c_int64, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, dp, ctypes.c_int]
        lib.kda_oracle_decode_step.restype = ctypes.c_int
        lib.kda_oracle_default_threads.restype = ctypes.c_int
        self.lib = lib

    def default_threads(self) -> int:
        return int(self.lib.kda_oracle_default_threads())

    def prefill(self, q, k, v, g, beta, S0, cu_seqlens, nthreads: int = 0):
        """Token-by-token prefill over a packed batch, in fp64.

        q, k, g: [T, H, dk]; v: [T, H, dv]; beta: [T, H]; S0: [N, H, dk, dv]
        or None (zeros); cu_seqlens: [N+1] offsets.  Returns (o [T, H, dv],
        S_T [N, H, dk, dv], threads used), all fp64 numpy arrays.
        """
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        cu = np.ascontiguousarray(np.asarray(
            cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
            dtype=np.int64))
        T, H, dk = q.shape
        dv = v.shape[2]
        N = cu.shape[0] - 1
        S0a = None if S0 is None else _f64(S0)
        o = np.zeros((T, H, dv), dtype=np.float64)
        S_T = np.zeros((N, H, dk, dv), dtype=np.float64)
        r = self.lib.kda_oracle_prefill(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(S0a),
            cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), N, T, H, dk, dv,
            _ptr(o), _ptr(S_T), int(nthreads))
        if r < 0:
            raise ValueError("kda_oracle_prefill rejected its arguments (%d)" % r)
        return o, S_T, r

    def decode_step(self, q, k, v, g, beta, S, nthreads: int = 0):
        """One decode step: every sequence consumes one token.

        q, k, g: [B, H, dk]; v: [B, H, dv]; beta: [B, H]; S: [B, H, dk, dv].
        Returns (o [B, H, dv], S' [B, H, dk, dv]) as fp64 arrays; S is not
        modified.
        """
        q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
        Sn = _f64(S).copy()
        B, H, dk = q.shape
        dv = v.shape[2]
        o = np.zeros((B, H, dv), dtype=np.float64)
        r = self.lib.kda_oracle_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(Sn), B, H,
            dk, dv, _ptr(o), int(nthreads))
        if r < 0:
            raise ValueError("kda_oracle_decode_step rejected its arguments (%d)" % r)
        return o, Sn


def _load() -> OracleLib:
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def _f64(x) -> np.ndarray:
    """Exact fp64 copy of a stored array (torch tensor or numpy array)."""
    if hasattr(x, "detach"):  # torch tensor: upcast exactly, then to numpy
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return _load().default_threads()


def prefill(q, k, v, g, beta, S0, cu_seqlens, nthreads: int = 0):
    """See :meth:`OracleLib.prefill` (default library)."""
    return _load().prefill(q, k, v, g, beta, S0, cu_seqlens, nthreads)


def decode_step(q, k, v, g, beta, S, nthreads: int = 0):
    """See :meth:`OracleLib.decode_step` (default library)."""
    return _load().decode_step(q, k, v, g, beta, S, nthreads)


def gdn_prefill(q, k, v, g, beta, S0, cu_seqlens, nthreads: int = 0):
    """Gated DeltaNet prefill: g is [T, H], one log-gate per head and token.

    The lineage essay's section "KDA: Kimi의 비법" describes KDA as Gated
    DeltaNet with its scalar alpha turned into a per-channel vector, so a
    scalar gate is the per-channel gate with every channel equal: g is
    broadcast over dk and the KDA recurrence runs unchanged.
    """
    g = _f64(g)
    dk = tuple(q.shape)[-1]
    gb = np.ascontiguousarray(np.broadcast_to(g[..., None], g.shape + (dk,)))
    return prefill(q, k, v, gb, beta, S0, cu_seqlens, nthreads)


def gdn_decode_step(q, k, v, g, beta, S, nthreads: int = 0):
    """Gated DeltaNet decode step: g is [B, H] (see :func:`gdn_prefill`)."""
    g = _f64(g)
    dk = tuple(q.shape)[-1]
    gb = np.ascontiguousarray(np.broadcast_to(g[..., None], g.shape + (dk,)))
    return decode_step(q, k, v, gb, beta, S, nthreads)
