"""The fp64 reverse-scan oracle over many (sequence, head) units in a pool of
worker processes (test infrastructure).

``oracle.chunked.chunked_bwd_dh`` is plain numpy and runs one unit at a time
in a single thread: a full-size workload (128 to 512 units of up to 65536
tokens) takes minutes that way.  The units are independent, so each worker
runs whole units on its own.  The pool starts its workers with ``spawn`` (a
process forked after the CUDA context exists can hang), and a worker imports
numpy and the oracle only: no torch, no CUDA library.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor

import numpy as np


def _run_unit(args):
    """Worker: one unit as a one-sequence, one-head problem, fp64."""
    from oracle import chunked as oc
    key, q, k, v, g, beta, scale, do, dv_in, dht = args
    f = lambda a: None if a is None else np.asarray(a, np.float64)  # noqa: E731
    dhck, dv2, dh0 = oc.chunked_bwd_dh(f(q), f(k), f(v), f(g), f(beta), scale, f(do), f(dv_in), dht=f(dht))
    return key, dhck[:, 0], dv2[0, :, 0], dh0[0, 0]


def unit_jobs(xn, gn, scale, units, starts, lens):
    """Per-unit argument tuples from numpy copies of the inputs (float32, which
    holds the bf16 / fp32 values exactly): xn = {q, k, v, g, beta} in the
    packed [rows, H, ...] layout, gn = {do, dv_in, dht}."""
    for s, h in units:
        a, n = starts[s], lens[s]
        sl = slice(a, a + n)
        one = lambda t: t[sl, h][None, :, None]  # noqa: E731  [1, n, 1, ...]
        dht = None if gn["dht"] is None else gn["dht"][s, h][None, None]
        yield ((s, h), one(xn["q"]), one(xn["k"]), one(xn["v"]), one(xn["g"]), xn["beta"][sl, h][None, :, None],
               scale, one(gn["do"]), one(gn["dv_in"]), dht)


def map_units(jobs, workers=None):
    """Yields (key, dhck [chunks, K, V], dv2 [n, V], dh0 [K, V]) per unit, in
    completion order, from a spawn pool."""
    n = workers or max(1, min(32, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                              else (os.cpu_count() or 1)))
    ctx = mp.get_context("spawn")
    with ProcessPoolExecutor(max_workers=n, mp_context=ctx) as ex:
        yield from ex.map(_run_unit, jobs, chunksize=1)
