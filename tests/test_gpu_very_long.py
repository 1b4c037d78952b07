"""One sequence four times longer than the long workload: 262 144 tokens
(4096 chunks) of two heads at K = V = 128, with the long workload's decay
(mu = 5, so the state keeps a long memory) and a random initial state.

The automatic plan scans it in many parallel segments (the map pass, the
chain of the segments' affine maps and the output pass); the single-pass
fused plan walks all 4096 chunks in one CTA per head.  Every element of o and
ht is compared with the fp64 token recurrence under the forward's
tolerances, and the figures are printed, so that the error's growth with the
length of the recurrence is on record.
"""
from __future__ import annotations

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import assert_within, compare, oracle_ref, report, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

W = synth.Workload("very_long", B=1, T=262144, H=2, K=128, V=128, mu=5.0, seed=20261213)


@pytest.fixture(scope="module")
def problem():
    x = synth.make_inputs(W)
    o_ref, ht_ref = oracle_ref(x)
    return x, o_ref, ht_ref


def _run(x, plan):
    d = to_dev(x)
    dims = kda.make_dims(W.B, W.T, W.H, W.K, W.V)
    ws = kda.new_workspace(dims, "cuda")
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws, plan=plan)
    torch.cuda.synchronize()
    assert kda.status(ws) == 0
    return o, ht, kda.workspace_layout(dims)


def test_automatic_plan(problem):
    x, o_ref, ht_ref = problem
    o, ht, lay = _run(x, None)
    assert lay.seg_count > 1  # the segmented scan
    res = compare(x, o, ht, o_ref, ht_ref)
    report(f"very long, {lay.seg_count} segments of {lay.seg_len} chunks", res)
    assert_within(res, "very long")


def test_fused_plan(problem):
    x, o_ref, ht_ref = problem
    o, ht, _ = _run(x, "fused")
    res = compare(x, o, ht, o_ref, ht_ref)
    report("very long, fused", res)
    assert_within(res, "very long fused")
