"""Tensors of more than 2^31 elements through the forward and the reverse
state scan.

The workload has B = 2 sequences of 65 573 tokens (a ragged last chunk) over
128 heads at K = V = 128, so q, k, v, o, do, dv_in and dv2 each hold
2.15e9 elements (4.3 GB, past every 32-bit element index) and g 8.6 GB (past
every 32-bit byte offset); the workspace is 19.5 GB.  Inputs are drawn on the
device by the seeded generator; the (sequence, head) units checked, among
them the last one (the largest offsets in every tensor), are copied back and
run through the fp64 oracle on their own.  Tolerances are the forward's.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gb300 import synth
from oracle import chunked as oc
from parity_util import MAXREL_O, REL_HT, REL_O

pytestmark = pytest.mark.gpu

W = synth.Workload("beyond_int32", B=2, T=65573, H=128, K=128, V=128, seed=20261211)
UNITS = [(1, 127), (0, 0), (1, 64)]


def _unit(x, b, h, names):
    """The inputs of (sequence b, head h) as a one-sequence, one-head problem on the CPU."""
    u = {}
    for n in names:
        t = x[n]
        if t is None:
            u[n] = None
        elif n in ("h0", "dht"):
            u[n] = t[b:b + 1, h:h + 1].cpu().contiguous()
        else:
            u[n] = t[b:b + 1, :, h:h + 1].cpu().contiguous()
    return u


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.fixture(scope="module")
def problem():
    import chunked_gated_delta_gb300 as kda
    free, _ = torch.cuda.mem_get_info()
    if free < 90e9:
        pytest.skip(f"needs ~75 GB of free device memory, {free / 1e9:.0f} GB free")
    x = synth.make_inputs_on(W, "cuda", with_bwd=True)
    assert x["q"].numel() > 2 ** 31 and x["g"].numel() * 4 > 2 ** 32
    dims = kda.make_dims(W.B, W.T, W.H, W.K, W.V)
    ws = kda.new_workspace(dims, "cuda")
    o, ht = kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"], workspace=ws)
    dhck, dv2, dh0 = kda.bwd_dh(x["scale"], x["do"], x["dv_in"], x["dht"], dims, ws)
    torch.cuda.synchronize()
    assert kda.status(ws) == 0
    yield x, o, ht, dhck, dv2, dh0
    del x, o, ht, dhck, dv2, dh0, ws
    torch.cuda.empty_cache()


def test_forward_beyond_int32_elements(problem):
    x, o, ht, *_ = problem
    for b, h in UNITS:
        u = _unit(x, b, h, ("q", "k", "v", "g", "beta", "h0"))
        o_ref, ht_ref = oracle.recurrent_fwd(u["q"], u["k"], u["v"], u["g"], u["beta"], x["scale"], h0=u["h0"])
        og = o[b, :, h].double().cpu().numpy()
        want = o_ref[0, :, 0]
        assert np.all(np.isfinite(og))
        assert _rel(og, want) <= REL_O, (b, h)
        assert np.max(np.abs(og - want)) <= MAXREL_O * np.max(np.abs(want)), (b, h)
        assert _rel(ht[b, h].double().cpu().numpy(), ht_ref[0, 0]) <= REL_HT, (b, h)


def test_reverse_scan_beyond_int32_elements(problem):
    x, _, _, dhck, dv2, dh0 = problem
    nt = (W.T + 63) // 64
    b, h = UNITS[0]  # the last unit: the largest offsets of dv2, the checkpoints and dh0
    u = _unit(x, b, h, ("q", "k", "v", "g", "beta", "do", "dv_in", "dht"))
    f = lambda t: t.double().numpy()  # noqa: E731
    ck_r, dv2_r, dh0_r = oc.chunked_bwd_dh(f(u["q"]), f(u["k"]), f(u["v"]), f(u["g"]), f(u["beta"]),
                                           x["scale"], f(u["do"]), f(u["dv_in"]), dht=f(u["dht"]))
    # checkpoints are [chunks, H, K, V] in chunk-table order: sequence b's chunks start at b * nt
    ck_g = dhck[b * nt:(b + 1) * nt, h].double().cpu().numpy()
    dv2_g = dv2[b, :, h].double().cpu().numpy()
    for got, want, what in ((ck_g, ck_r[:, 0], "dhck"), (dv2_g, dv2_r[0, :, 0], "dv2"),
                            (dh0[b, h].double().cpu().numpy(), dh0_r[0, 0], "dh0")):
        assert np.all(np.isfinite(got)), what
        assert _rel(got, want) <= REL_O, what
        assert np.max(np.abs(got - want)) <= MAXREL_O * np.max(np.abs(want)), what
