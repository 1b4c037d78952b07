"""ctypes binding of ``libkda.so`` (the C ABI in ``include/kda.h``).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  There
is no CPU fallback: if the library cannot be loaded, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

KDA_OK = 0
STATUS_NAMES = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_ALIGNMENT",
    4: "KDA_ERR_WORKSPACE", 5: "KDA_ERR_CUDA", 6: "KDA_ERR_TIMEOUT", 7: "KDA_ERR_BAD_SEQLENS",
}

# Every symbol the header declares (checked by the CPU test suite).
EXPORTS = ("kda_fwd_workspace_size", "kda_fwd", "kda_fwd_intra", "kda_fwd_scan", "kda_fwd_status",
           "kda_status_string", "kda_chunk_table", "kda_workspace_layout", "kda_fwd_host_arena_size",
           "kda_fwd_host", "kda_fwd_noalloc", "kda_selftest_wait_timeout", "kda_bwd_dh",
           "kda_fwd_ex", "kda_fwd_intra_ex", "kda_fwd_scan_ex", "kda_bwd_dh_ex", "kda_fwd_state_map",
           "kda_chain_states")


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = code
        msg = status_string(code) if _lib is not None else STATUS_NAMES.get(code, str(code))
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({msg})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("K", ctypes.c_int32), ("V", ctypes.c_int32), ("num_seqs", ctypes.c_int32)]


class FwdOpts(ctypes.Structure):
    """kda_fwd_opts: interface variants of the forward (all zero = kda_fwd)."""
    _fields_ = [("io_dtype", ctypes.c_int32), ("state_dtype", ctypes.c_int32),
                ("beta_logits", ctypes.c_int32), ("qk_heads", ctypes.c_int32), ("plan", ctypes.c_int32)]


IO_BF16, IO_F16 = 0, 1
STATE_F32, STATE_BF16 = 0, 1
PLAN_AUTO, PLAN_TWO_STAGE, PLAN_FUSED = 0, 1, 2
PLANS = {None: PLAN_AUTO, "auto": PLAN_AUTO, "two_stage": PLAN_TWO_STAGE, "fused": PLAN_FUSED}


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("status", "seq_info", "chunk_info", "gd", "qg", "kg", "w", "u", "aqk", "total")] + [
        ("max_chunks", ctypes.c_int32), ("chunk", ctypes.c_int32),
        ("seg_count", ctypes.c_int32), ("seg_len", ctypes.c_int32),
        ("pq", ctypes.c_size_t), ("hin", ctypes.c_size_t),
        ("stage_count", ctypes.c_int32), ("stage_len", ctypes.c_int32)]


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libkda.so (building it in-tree with nvcc first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            if not build_if_missing:
                raise RuntimeError(f"{path} is missing; run chunked_gated_delta_gb300.build.build()")
            _build.build()
        lib = ctypes.CDLL(path)
        P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        D = ctypes.POINTER(Dims)
        O = ctypes.POINTER(FwdOpts)
        sig = {
            "kda_fwd_workspace_size": (SZ, [D]),
            "kda_fwd": (ctypes.c_int, [P, P, P, P, P, F32, P, P, P, P, D, P, SZ, P]),
            "kda_fwd_intra": (ctypes.c_int, [P, P, P, P, P, P, D, P, SZ, P]),
            "kda_fwd_scan": (ctypes.c_int, [F32, P, P, P, D, P, SZ, P]),
            "kda_fwd_status": (ctypes.c_int, [P, P]),
            "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "kda_chunk_table": (I32, [P, I32, I32, P, P]),
            "kda_workspace_layout": (ctypes.c_int, [D, ctypes.POINTER(WsLayout)]),
            "kda_fwd_host_arena_size": (SZ, [D]),
            "kda_fwd_host": (ctypes.c_int, [P, P, P, P, P, F32, P, P, P, P, D, P, SZ, P]),
            "kda_fwd_noalloc": (ctypes.c_int, [P, P, P, P, P, F32, P, P, P, P, D, P]),
            "kda_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_ulonglong, P]),
            "kda_bwd_dh": (ctypes.c_int, [F32, P, P, P, P, P, P, D, P, SZ, P]),
            "kda_fwd_ex": (ctypes.c_int, [P, P, P, P, P, F32, P, P, P, P, D, O, P, SZ, P]),
            "kda_fwd_intra_ex": (ctypes.c_int, [P, P, P, P, P, P, D, O, P, SZ, P]),
            "kda_fwd_scan_ex": (ctypes.c_int, [F32, P, P, P, D, O, P, SZ, P]),
            "kda_bwd_dh_ex": (ctypes.c_int, [F32, P, P, P, P, P, P, D, O, P, SZ, P]),
            "kda_fwd_state_map": (ctypes.c_int, [P, P, P, P, P, P, P, D, P, SZ, P]),
            "kda_chain_states": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, I32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def status_string(code: int) -> str:
    return load_library().kda_status_string(int(code)).decode()


def make_dims(B, T, H, K, V, num_seqs=0) -> Dims:
    return Dims(int(B), int(T), int(H), int(K), int(V), int(num_seqs))


def workspace_size(dims: Dims) -> int:
    return int(load_library().kda_fwd_workspace_size(ctypes.byref(dims)))


def workspace_layout(dims: Dims) -> WsLayout:
    out = WsLayout()
    rc = load_library().kda_workspace_layout(ctypes.byref(dims), ctypes.byref(out))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_workspace_layout")
    return out


def chunk_table(cu_seqlens, chunk: int = 64):
    """Host chunk table: (tile_base list, t_tiles list, total) or raises ValueError."""
    lib = load_library()
    cu = [int(x) for x in cu_seqlens]
    n = len(cu) - 1
    if n < 0:
        raise ValueError("cu_seqlens must have at least one entry")
    cu_a = (ctypes.c_int32 * len(cu))(*cu)
    tb = (ctypes.c_int32 * max(n, 1))()
    tt = (ctypes.c_int32 * max(n, 1))()
    total = lib.kda_chunk_table(cu_a, n, int(chunk), tb, tt)
    if total < 0:
        raise ValueError("invalid cu_seqlens / chunk")
    return list(tb)[:n], list(tt)[:n], int(total)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc, where):
    if rc != KDA_OK:
        raise KdaError(rc, where)


def _dims_of(q, v, cu_seqlens):
    B, T, _, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    N = 0 if cu_seqlens is None else cu_seqlens.numel() - 1
    return make_dims(B, T, H, K, V, N), (B if cu_seqlens is None else N)


def _check_inputs(q, k, v, g, beta, h0, cu_seqlens):
    import torch
    io = q.dtype if q.dtype in (torch.bfloat16, torch.float16) else torch.bfloat16
    for name, t, dt in (("q", q, io), ("k", k, io), ("v", v, io), ("g", g, torch.float32), ("beta", beta, io)):
        if t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {dt}")
    if k.shape != q.shape:
        raise TypeError("q and k must have the same shape")
    if h0 is not None and (h0.dtype not in (torch.float32, torch.bfloat16) or not h0.is_cuda
                           or not h0.is_contiguous()):
        raise TypeError("h0 must be a contiguous CUDA float32 or bfloat16 tensor")
    if cu_seqlens is not None and (cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda):
        raise TypeError("cu_seqlens must be a CUDA int32 tensor")


def new_workspace(dims: Dims, device):
    import torch
    n = workspace_size(dims)
    if n == 0:
        raise KdaError(1, "kda_fwd_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def fwd(q, k, v, g, beta, scale=None, h0=None, cu_seqlens=None, output_final_state=True,
        workspace=None, out=None, final_state=None, stream=None, beta_logits=False, state_dtype=None,
        plan=None):
    """KDA chunked forward on the GPU.  Returns (o, ht) (ht None if not requested).

    q, k: [B,T,Hqk,K]; v: [B,T,H,V]; beta: [B,T,H], all bf16 or all fp16 (o
    follows); g: fp32 [B,T,H,K] (natural-log decay); h0: [N,H,K,V] fp32 or bf16
    or None; cu_seqlens: int32 [N+1] on the device (B must be 1) or None.
    H must be a multiple of Hqk (grouped value heads: value head h reads q/k
    head h // (H // Hqk)).  ``beta_logits``: beta holds logits, the kernel
    applies the sigmoid.  ``state_dtype`` (torch.float32 / torch.bfloat16) of ht;
    defaults to h0's dtype, else fp32.  ``workspace`` (uint8 CUDA tensor) may be
    passed to avoid an allocation per call.  ``plan``: None / "auto" /
    "two_stage" (the two kernels; the workspace keeps the intermediates for
    bwd_dh) or "fused" (the single-pass kernel: bf16 I/O, fp32 state, activated
    beta, equal heads).
    """
    import torch
    _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    lib = load_library()
    dims, N = _dims_of(q, v, cu_seqlens)
    B, T, Hqk, K = q.shape
    H, V = v.shape[2], v.shape[-1]
    if scale is None:
        scale = K ** -0.5
    if state_dtype is None:
        state_dtype = h0.dtype if h0 is not None else torch.float32
    if h0 is not None and h0.dtype != state_dtype:
        raise TypeError("h0 and ht must have the same dtype")
    if plan not in PLANS:
        raise ValueError(f"plan must be one of {sorted(k for k in PLANS if k)}")
    opts = FwdOpts(IO_F16 if q.dtype == torch.float16 else IO_BF16,
                   STATE_BF16 if state_dtype == torch.bfloat16 else STATE_F32,
                   1 if beta_logits else 0, Hqk if Hqk != H else 0, PLANS[plan])
    if workspace is None:
        workspace = new_workspace(dims, q.device)
    o = out if out is not None else torch.empty((B, T, H, V), dtype=q.dtype, device=q.device)
    ht = None
    if output_final_state:
        ht = final_state if final_state is not None else torch.empty((N, H, K, V), dtype=state_dtype,
                                                                      device=q.device)
    rc = lib.kda_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale), _ptr(h0),
                        _ptr(cu_seqlens), _ptr(o), _ptr(ht), ctypes.byref(dims), ctypes.byref(opts),
                        _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "kda_fwd_ex")
    return o, ht


def fwd_intra(q, k, v, g, beta, cu_seqlens, dims: Dims, workspace, stream=None):
    rc = load_library().kda_fwd_intra(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens),
                                      ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                                      _stream_handle(stream))
    _check(rc, "kda_fwd_intra")


def fwd_scan(scale, h0, o, ht, dims: Dims, workspace, stream=None):
    rc = load_library().kda_fwd_scan(float(scale), _ptr(h0), _ptr(o), _ptr(ht), ctypes.byref(dims),
                                     _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(rc, "kda_fwd_scan")


def state_map(q, k, v, g, beta, cu_seqlens=None, workspace=None, stream=None):
    """kda_fwd_state_map: the affine state map [P | Q] (fp32 [N, H, K, K + V])
    of these tokens of every (sequence, head).  Returns (pq, workspace, dims);
    the workspace keeps the intra-chunk intermediates for fwd_scan."""
    import torch
    _check_inputs(q, k, v, g, beta, None, cu_seqlens)
    if q.dtype != torch.bfloat16 or q.shape[2] != v.shape[2]:
        raise TypeError("state_map takes the default interface (bf16 I/O, equal heads)")
    dims, N = _dims_of(q, v, cu_seqlens)
    K, V, H = q.shape[-1], v.shape[-1], v.shape[2]
    if workspace is None:
        workspace = new_workspace(dims, q.device)
    pq = torch.empty((N, H, K, K + V), dtype=torch.float32, device=q.device)
    rc = load_library().kda_fwd_state_map(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(cu_seqlens), _ptr(pq),
                                          ctypes.byref(dims), _ptr(workspace), workspace.numel(),
                                          _stream_handle(stream))
    _check(rc, "kda_fwd_state_map")
    return pq, workspace, dims


def chain_states(pq_all, h0=None, stream=None):
    """kda_chain_states: entry states h_in [R, N, H, K, V] of R consecutive token
    ranges from their gathered maps pq_all [R, N, H, K, K + V] (fp32, CUDA)."""
    import torch
    if pq_all.dtype != torch.float32 or not pq_all.is_cuda or not pq_all.is_contiguous() or pq_all.dim() != 5:
        raise TypeError("pq_all must be a contiguous CUDA float32 tensor [R, N, H, K, K + V]")
    R, N, H, K, KV = pq_all.shape
    V = KV - K
    if h0 is not None and (h0.dtype != torch.float32 or not h0.is_cuda or not h0.is_contiguous()
                           or tuple(h0.shape) != (N, H, K, V)):
        raise TypeError("h0 must be a contiguous CUDA float32 tensor [N, H, K, V]")
    h_in = torch.empty((R, N, H, K, V), dtype=torch.float32, device=pq_all.device)
    rc = load_library().kda_chain_states(_ptr(pq_all), _ptr(h0), _ptr(h_in), R, N, H, K, V, _stream_handle(stream))
    _check(rc, "kda_chain_states")
    return h_in


def status(workspace, stream=None) -> int:
    """Synchronise the stream and return the kernels' recorded status code."""
    return int(load_library().kda_fwd_status(_ptr(workspace), _stream_handle(stream)))


def exact_path_tiles(workspace, dims: Dims, stream=None) -> int:
    """Synchronise the stream and return the diagnostic count of (chunk, head)
    tiles whose gated sums took the exact per-element path in the last
    forward on this workspace (the int32 after the status word)."""
    import torch
    status(workspace, stream)
    off = workspace_layout(dims).status + 4
    return int(workspace[off:off + 4].cpu().view(torch.int32).item())


def host_arena_size(dims: Dims) -> int:
    return int(load_library().kda_fwd_host_arena_size(ctypes.byref(dims)))


def fwd_host(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, dims: Dims, arena, stream=None):
    """kda_fwd_host: all tensors are (preferably pinned) CPU tensors; ``arena`` is a
    uint8 CUDA tensor of at least host_arena_size(dims) bytes.  Asynchronous on
    ``stream``; synchronise before reading o / ht."""
    rc = load_library().kda_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                     _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(ht), ctypes.byref(dims),
                                     _ptr(arena), arena.numel(), _stream_handle(stream))
    _check(rc, "kda_fwd_host")


NOALLOC_SCRATCH_BYTES = 64 << 20  # KDA_NOALLOC_SCRATCH_BYTES in include/kda.h


def fwd_noalloc(q, k, v, g, beta, scale, h0, cu_seqlens, o, ht, stream=None):
    """kda_fwd_noalloc: the forward with the library's built-in scratch array as
    workspace (no device allocation by the library).  All tensors are CUDA
    tensors allocated by the caller; o and ht are written in place."""
    import torch
    _check_inputs(q, k, v, g, beta, h0, cu_seqlens)
    if q.dtype != torch.bfloat16 or q.shape[2] != v.shape[2] or (h0 is not None and h0.dtype != torch.float32):
        raise TypeError("kda_fwd_noalloc takes the default interface (bf16 I/O, fp32 state, equal heads)")
    dims, _ = _dims_of(q, v, cu_seqlens)
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    rc = load_library().kda_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), float(scale),
                                        _ptr(h0), _ptr(cu_seqlens), _ptr(o), _ptr(ht),
                                        ctypes.byref(dims), _stream_handle(stream))
    _check(rc, "kda_fwd_noalloc")


def selftest_wait_timeout(limit_ns: int = 1_000_000, stream=None) -> int:
    """Run the bounded-wait self-check; returns the status code (6 = timed out as designed)."""
    import torch
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    return int(load_library().kda_selftest_wait_timeout(_ptr(word), int(limit_ns), _stream_handle(stream)))


def bwd_dh(scale, do, dv_in, dht, dims: Dims, workspace, want_dhck=True, want_dh0=True, stream=None,
           state_dtype=None):
    """Reverse state scan on the GPU (kda_bwd_dh_ex).  ``workspace`` must hold
    the intra-chunk intermediates of the same inputs (from fwd / fwd_intra).
    do, dv_in: [B,T,H,V] bf16 or fp16 (dv2 follows); dht: [N,H,K,V] fp32 or
    bf16 or None (dh0 follows it, or ``state_dtype``).  Returns (dhck
    [max_chunks,H,K,V] bf16 or None, dv2 [B,T,H,V], dh0 [N,H,K,V] or None)."""
    import torch
    io = do.dtype
    if io not in (torch.bfloat16, torch.float16):
        raise TypeError("do must be bf16 or fp16")
    for name, t in (("do", do), ("dv_in", dv_in)):
        if t.dtype != io or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous CUDA tensor of dtype {io}")
    if state_dtype is None:
        state_dtype = dht.dtype if dht is not None else torch.float32
    if state_dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("the state dtype is float32 or bfloat16")
    if dht is not None and (dht.dtype != state_dtype or not dht.is_cuda or not dht.is_contiguous()):
        raise TypeError("dht must be a contiguous CUDA tensor of the state dtype")
    B, T, H, V = do.shape
    K = dims.K
    N = dims.num_seqs if dims.num_seqs > 0 else dims.B
    lay = workspace_layout(dims)
    dev = do.device
    dhck = torch.empty((lay.max_chunks, H, K, V), dtype=torch.bfloat16, device=dev) if want_dhck else None
    dv2 = torch.zeros((B, T, H, V), dtype=io, device=dev)
    dh0 = torch.empty((N, H, K, V), dtype=state_dtype, device=dev) if want_dh0 else None
    opts = FwdOpts(IO_F16 if io == torch.float16 else IO_BF16,
                   STATE_BF16 if state_dtype == torch.bfloat16 else STATE_F32, 0, 0)
    rc = load_library().kda_bwd_dh_ex(float(scale), _ptr(do), _ptr(dv_in), _ptr(dht), _ptr(dhck), _ptr(dv2),
                                      _ptr(dh0), ctypes.byref(dims), ctypes.byref(opts), _ptr(workspace),
                                      workspace.numel(), _stream_handle(stream))
    _check(rc, "kda_bwd_dh_ex")
    return dhck, dv2, dh0
