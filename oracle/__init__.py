"""fp64 CPU oracle for the KDA forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  It shares no code with the CUDA
library (``chunked_gated_delta_gb300``) and never imports it.

Two independent references live here:

* :func:`recurrent_fwd` -- the token-by-token KDA recurrence in fp64, written in
  plain C (``kda_oracle.c``) and threaded over (sequence, head) units.  This is
  the definition every GPU result is compared against.
* :mod:`oracle.chunked` -- the chunked form (in-chunk cumsum, gated Aqk, the
  beta-weighted lower-triangular system, w/u, and the inter-chunk scan) in
  fp64 numpy, used to pin the recurrence and to check GPU intermediates.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, invariants, hand-worked fixtures and the chunked-vs-recurrent
agreement); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` into ``libkda_oracle.so`` next to it (gcc, -O2)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I = ctypes.c_int
            for name in ("kda_oracle_fwd_f64", "kda_oracle_fwd_bf16"):
                fn = getattr(lib, name)
                fn.restype = I
                fn.argtypes = [P, P, P, P, P, ctypes.c_double, P, P, I, I, I, I, P, I, P, P, I]
            _lib = lib
    return _lib


def default_threads(units: int | None = None) -> int:
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    n = max(1, int(n or 1))
    return n if units is None else max(1, min(n, units))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bits16(x):
    """A bf16 array given as torch bf16 / numpy uint16 bit patterns -> uint16 numpy."""
    if hasattr(x, "dtype") and str(getattr(x, "dtype", "")) == "torch.bfloat16":
        import torch  # only to reinterpret bits; no arithmetic
        return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))
    a = np.ascontiguousarray(x)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs must be torch.bfloat16 or uint16 bit patterns")
    return a


def _np(x, dtype):
    if hasattr(x, "numpy") and not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=dtype)


def recurrent_fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, units=None,
                  want_ht=True, nthreads=None, fp64_inputs=False):
    """Token-by-token KDA recurrence in fp64.

    Shapes: q, k, g ``[B, T, H, K]``; v ``[B, T, H, V]``; beta ``[B, T, H]``;
    h0 ``[N, H, K, V]`` or None.  Without ``cu_seqlens`` the N = B batch rows are
    the sequences; with ``cu_seqlens`` (int, ``[N+1]``) B must be 1 and the
    sequences are its slices.

    ``fp64_inputs=False`` (default): q, k, v, beta are bf16 (torch bf16 or
    uint16 bits) and g, h0 fp32 -- the GPU path's storage formats, widened
    exactly.  ``fp64_inputs=True``: every input is taken as float64 as given.

    ``units``: optional list of (sequence, head) pairs to compute; other rows of
    ``o`` are left as NaN.  Returns ``(o [B,T,H,V] float64, ht [N,H,K,V] float64
    or None)``.
    """
    lib = _load()
    if fp64_inputs:
        qa, ka, va, ga, ba = (_np(x, np.float64) for x in (q, k, v, g, beta))
        ha = None if h0 is None else _np(h0, np.float64)
        fn = lib.kda_oracle_fwd_f64
    else:
        qa, ka, va, ba = (_bits16(x) for x in (q, k, v, beta))
        ga = _np(g, np.float32)
        ha = None if h0 is None else _np(h0, np.float32)
        fn = lib.kda_oracle_fwd_bf16
    B, T, H, K = qa.shape
    V = va.shape[-1]
    if cu_seqlens is None:
        N = B
        cu = (np.arange(B + 1, dtype=np.int64) * T).astype(np.int32)
    else:
        if B != 1:
            raise ValueError("cu_seqlens requires B == 1")
        cu = _np(cu_seqlens, np.int64).astype(np.int32)
        N = cu.shape[0] - 1
    if ha is not None and ha.shape != (N, H, K, V):
        raise ValueError(f"h0 shape {ha.shape} != {(N, H, K, V)}")
    o = np.full((B, T, H, V), np.nan, dtype=np.float64)
    ht = np.zeros((N, H, K, V), dtype=np.float64) if want_ht else None
    if units is None:
        ua, nu = None, N * H
    else:
        ua = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        nu = ua.shape[0]
    nth = default_threads(nu) if nthreads is None else int(nthreads)
    rc = fn(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ga), _ptr(ba), float(scale), _ptr(ha),
            _ptr(cu), N, H, K, V, _ptr(ua), nu, _ptr(o), _ptr(ht), nth)
    if rc != 0:
        raise RuntimeError(f"kda oracle failed with code {rc}")
    return o, ht
