"""Chunked KDA forward in fp64 numpy -- TEST INFRASTRUCTURE (see oracle/__init__).

This is the chunkwise algorithm that the GPU path implements, written step by
step in the notation of kernel-fun ``kda/_kernels/fwd_state.py`` (module
docstring: the intra-stage operands ``qg``, ``kg``, ``Aqk``, ``w``, ``u``, the
per-chunk decay vector ``G`` = last row of ``g2``, and the per-chunk scan
``WH = w@h; v' = u - WH; o = scale*qg@h + Aqk@v'; h <- exp2(G)*h + kg^T@v'``).
The two operands that fwd_state.py consumes but does not define, ``w`` and
``u``, follow from the per-token recurrence: with the inclusive in-chunk decay
gamma_i = exp2(g2_i),

    A[i, j] = beta_i * sum_d k_id k_jd exp2(g2_id - g2_jd)      (j < i, else 0)
    T       = (I + A)^-1                                          (unit lower triangular)
    w       = T diag(beta) (k * exp2(g2)),   u = T diag(beta) v

so that v' = u - w @ h is the chunk's vector of delta-rule corrections.
FlashKDA (the "KDA源码剖析之FlashKDA（下）" walk-through, its INV operand) uses the
same inverse at chunk 16.

No blocking or reassociation is done beyond what these equations state: every
gate factor is an explicit exp2 of a difference, so nothing overflows for any
finite decay.  A tail chunk (sequence length not a multiple of C) is padded
with inert rows (q = k = v = 0, g = 0, beta = 0), which leaves the recurrence
over the valid rows unchanged.
"""
from __future__ import annotations

import numpy as np

LOG2E = 1.0 / np.log(2.0)


def _pad_rows(x, C):
    n = x.shape[0]
    r = (-n) % C
    if r == 0:
        return x
    pad = np.zeros((r,) + x.shape[1:], dtype=x.dtype)
    return np.concatenate([x, pad], axis=0)


def chunk_intra(q, k, v, g, beta, scale, C=64):
    """Intra-chunk stage for one (sequence, head).

    q, k, g: [L, K]; v: [L, V]; beta: [L] (fp64).  Returns a list (one entry per
    chunk) of dicts with keys ``g2`` [C,K] (log2-space inclusive cumsum),
    ``G`` [K], ``qg``, ``kg`` [C,K], ``Aqk`` [C,C] (scale folded in, zero above
    the diagonal), ``A`` [C,C] (strictly lower), ``T`` [C,C], ``w`` [C,K],
    ``u`` [C,V], ``valid`` (number of real rows).
    """
    L = q.shape[0]
    q, k, v, g = (_pad_rows(np.asarray(x, np.float64), C) for x in (q, k, v, g))
    beta = _pad_rows(np.asarray(beta, np.float64), C)
    out = []
    for c0 in range(0, q.shape[0], C):
        sl = slice(c0, c0 + C)
        qc, kc, vc, gc, bc = q[sl], k[sl], v[sl], g[sl], beta[sl]
        g2 = np.cumsum(gc, axis=0) * LOG2E           # chunk-local cumsum / ln2
        G = g2[-1].copy()                            # padded rows carry g = 0
        lower_eq = np.tril(np.ones((C, C), dtype=bool))       # j <= i
        lower = np.tril(np.ones((C, C), dtype=bool), k=-1)    # j < i
        # gate[i, j, d] = exp2(g2_id - g2_jd), only where it is used (j <= i)
        diff = g2[:, None, :] - g2[None, :, :]
        diff = np.where(lower_eq[:, :, None], diff, -np.inf)
        gate = np.exp2(diff)
        Aqk = scale * np.einsum("id,jd,ijd->ij", qc, kc, gate)
        Akk = np.einsum("id,jd,ijd->ij", kc, kc, gate)
        A = np.where(lower, bc[:, None] * Akk, 0.0)
        T = np.linalg.inv(np.eye(C) + A)
        w = T @ (bc[:, None] * (kc * np.exp2(g2)))
        u = T @ (bc[:, None] * vc)
        qg = qc * np.exp2(g2)
        kg = kc * np.exp2(G[None, :] - g2)
        out.append(dict(g2=g2, G=G, qg=qg, kg=kg, Aqk=Aqk, A=A, T=T, w=w, u=u,
                        valid=min(C, L - c0)))
    return out


def chunk_scan(chunks, h0, scale):
    """Inter-chunk state scan for one (sequence, head).

    ``chunks`` from :func:`chunk_intra`; h0 [K, V].  Returns (o [L, V], ht [K, V]).
    """
    h = np.array(h0, dtype=np.float64, copy=True)
    outs = []
    for ch in chunks:
        WH = ch["w"] @ h
        vp = ch["u"] - WH
        o = scale * (ch["qg"] @ h) + ch["Aqk"] @ vp
        h = np.exp2(ch["G"])[:, None] * h + ch["kg"].T @ vp
        outs.append(o[: ch["valid"]])
    V = h.shape[1]
    o = np.concatenate(outs, axis=0) if outs else np.zeros((0, V))
    return o, h


def chunked_fwd(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, C=64):
    """Chunked KDA forward over all sequences and heads, fp64.

    Same shapes and sequence conventions as :func:`oracle.recurrent_fwd`; the
    inputs are numpy arrays already in float64 (or anything numpy converts).
    Returns (o [B,T,H,V], ht [N,H,K,V]).
    """
    q, k, v, g, beta = (np.asarray(x, np.float64) for x in (q, k, v, g, beta))
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        cu = np.arange(B + 1) * T
        N = B
        flat = lambda x: x.reshape((B * T,) + x.shape[2:])  # noqa: E731
    else:
        assert B == 1
        cu = np.asarray(cu_seqlens, np.int64)
        N = len(cu) - 1
        flat = lambda x: x[0]  # noqa: E731
    qf, kf, vf, gf, bf = (flat(x) for x in (q, k, v, g, beta))
    o = np.zeros((B * T, H, V))
    ht = np.zeros((N, H, K, V))
    for s in range(N):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            h0sh = np.zeros((K, V)) if h0 is None else np.asarray(h0, np.float64)[s, h]
            if b == a:
                ht[s, h] = h0sh
                continue
            chunks = chunk_intra(qf[a:b, h], kf[a:b, h], vf[a:b, h], gf[a:b, h], bf[a:b, h],
                                 scale, C)
            os_, hs = chunk_scan(chunks, h0sh, scale)
            o[a:b, h] = os_
            ht[s, h] = hs
    return o.reshape(B, T, H, V), ht


def chunk_bwd_dh(chunks, do, dv_in, dht, scale):
    """Reverse state scan of the chunked forward for one (sequence, head), fp64.

    The backward companion of :func:`chunk_scan` in kernel-fun
    ``kda/_kernels/bwd_dhu.py`` (module docstring): with dh the gradient of the
    loss with respect to the state after the chunk being processed, chunks
    newest first,

        dhck[c] = dh                                  (checkpoint, before the update)
        dv2     = kg @ dh + dv_in                     (gradient w.r.t. v' of the chunk)
        dh      = exp2(G) * dh + scale qg^T @ do - w^T @ dv2
        dh0     = dh after the oldest chunk

    ``chunks`` from :func:`chunk_intra` (fp64 qg, kg, w, G; qg without scale);
    do, dv_in: [L, V]; dht: [K, V] (or None = zeros).  Returns (dhck [n_chunks,
    K, V], dv2 [L, V], dh0 [K, V]).  dv_in carries the chunk-local part of the
    v' gradient (the Aqk^T do term), which the dh scan takes as an input.
    """
    C = chunks[0]["qg"].shape[0] if chunks else 64
    K = chunks[0]["kg"].shape[1] if chunks else (dht.shape[0] if dht is not None else 0)
    V = do.shape[1]
    L = do.shape[0]
    do_p = _pad_rows(np.asarray(do, np.float64), C)
    dvi_p = _pad_rows(np.asarray(dv_in, np.float64), C)
    dh = np.zeros((K, V)) if dht is None else np.array(dht, dtype=np.float64, copy=True)
    dhck = np.zeros((len(chunks), K, V))
    dv2 = np.zeros((len(chunks) * C, V))
    for c in range(len(chunks) - 1, -1, -1):
        ch = chunks[c]
        sl = slice(c * C, (c + 1) * C)
        dhck[c] = dh
        d2 = ch["kg"] @ dh + dvi_p[sl]
        d2[ch["valid"]:] = 0.0  # padding rows are not part of the sequence
        dv2[sl] = d2
        dh = np.exp2(ch["G"])[:, None] * dh + scale * (ch["qg"].T @ do_p[sl]) - ch["w"].T @ d2
    return dhck, dv2[:L], dh


def scan_with_vprime(chunks, h0, scale, override=None):
    """The inter-chunk scan with an optional additive perturbation of one
    chunk's v' (``override = (c, dV)``); returns (o [L, V], ht [K, V]).  Used
    to check the backward's dv2 by finite differences of the forward."""
    h = np.array(h0, dtype=np.float64, copy=True)
    outs = []
    for c, ch in enumerate(chunks):
        vp = ch["u"] - ch["w"] @ h
        if override is not None and override[0] == c:
            vp = vp + override[1]
        o = scale * (ch["qg"] @ h) + ch["Aqk"] @ vp
        h = np.exp2(ch["G"])[:, None] * h + ch["kg"].T @ vp
        outs.append(o[: ch["valid"]])
    return np.concatenate(outs, axis=0), h


def chunked_bwd_dh(q, k, v, g, beta, scale, do, dv_in, h0=None, dht=None, cu_seqlens=None, C=64,
                   units=None):
    """Reverse state scan over all sequences and heads, fp64 (shapes as the
    forward; do, dv_in [B,T,H,V]; dht [N,H,K,V] or None).  Returns
    (dhck [total chunks, H, K, V] in chunk-table order, dv2 [B,T,H,V],
    dh0 [N,H,K,V]).  ``units`` (a list of (sequence, head)) restricts the work
    to those units; every other entry of the results is NaN."""
    q, k, v, g, beta, do, dv_in = (np.asarray(x, np.float64) for x in (q, k, v, g, beta, do, dv_in))
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is None:
        cu = np.arange(B + 1) * T
        N = B
        flat = lambda x: x.reshape((B * T,) + x.shape[2:])  # noqa: E731
    else:
        assert B == 1
        cu = np.asarray(cu_seqlens, np.int64)
        N = len(cu) - 1
        flat = lambda x: x[0]  # noqa: E731
    qf, kf, vf, gf, bf, dof, dvf = (flat(x) for x in (q, k, v, g, beta, do, dv_in))
    lens = np.diff(cu)
    tiles = (lens + C - 1) // C
    base = np.concatenate([[0], np.cumsum(tiles)])
    fill = 0.0 if units is None else np.nan
    dhck = np.full((int(base[-1]), H, K, V), fill)
    dv2 = np.full((B * T, H, V), fill)
    dh0 = np.full((N, H, K, V), fill)
    todo = [(s, h) for s in range(N) for h in range(H)] if units is None else list(units)
    for s, h in todo:
        a, b = int(cu[s]), int(cu[s + 1])
        dhts = None if dht is None else np.asarray(dht, np.float64)[s, h]
        if b == a:
            dh0[s, h] = 0.0 if dhts is None else dhts
            continue
        chunks = chunk_intra(qf[a:b, h], kf[a:b, h], vf[a:b, h], gf[a:b, h], bf[a:b, h], scale, C)
        # the scan's qg enters o with scale applied outside; chunk_intra's Aqk has scale inside
        ck, d2, d0 = chunk_bwd_dh(chunks, dof[a:b, h], dvf[a:b, h], dhts, scale)
        dhck[base[s]:base[s + 1], h] = ck
        dv2[a:b, h] = d2
        dh0[s, h] = d0
    return dhck, dv2.reshape(B, T, H, V), dh0
