"""Seeded random sweep of shapes and options through the forward (and the
reverse scan), each case checked against the fp64 oracle with the default
tolerances.  Covers combinations the targeted tests do not enumerate: odd
lengths, many short or empty sequences, head counts that change the scan's
kernel shape, the segmented plan, and the interface options together."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import assert_within, make, to_dev
from test_gpu_variants import errors, oracle_variant

pytestmark = pytest.mark.gpu

N_CASES = 24


def _case(i):
    rng = np.random.default_rng(7000 + i)
    K = int(rng.choice([64, 128]))
    V = int(rng.choice([64, 128]))
    Hqk = int(rng.choice([1, 2, 3]))
    H = Hqk * int(rng.choice([1, 2, 4]))
    io = torch.float16 if rng.random() < 0.3 else torch.bfloat16
    state = torch.bfloat16 if rng.random() < 0.3 else torch.float32
    logits = bool(rng.random() < 0.3)
    mu = float(rng.choice([3.0, 0.0, -4.0]))
    if rng.random() < 0.5:
        n = int(rng.integers(1, 9))
        lengths = [int(v) for v in rng.integers(0, 1500, size=n)]
        if rng.random() < 0.3:
            lengths[int(rng.integers(0, n))] = 0
        if sum(lengths) == 0:
            lengths[0] = 1
        w = make(T=0, H=H, K=K, V=V, mu=mu, seed=8000 + i)
        x = synth.make_variant_inputs(w, io_dtype=io, qk_heads=Hqk, beta_logits=logits, state_dtype=state,
                                      lengths=lengths)
    else:
        B = int(rng.integers(1, 4))
        T = int(rng.integers(1, 2500))
        w = make(B=B, T=T, H=H, K=K, V=V, mu=mu, seed=8000 + i)
        x = synth.make_variant_inputs(w, io_dtype=io, qk_heads=Hqk, beta_logits=logits, state_dtype=state)
    return x


@pytest.mark.parametrize("i", range(N_CASES))
def test_forward_random_case(i):
    from test_gpu_variants import run_variant
    x = _case(i)
    o, ht = run_variant(x)
    o_ref, ht_ref = oracle_variant(x)
    assert_within(errors(x, o, ht, o_ref, ht_ref), f"case {i}")


@pytest.mark.parametrize("i", range(0, N_CASES, 3))
def test_reverse_scan_random_case(i):
    """Every third case of the sweep through the reverse scan, with gradients in
    the case's io dtype and state in its state dtype."""
    from test_gpu_bwd import _dims, assert_bwd_within, compare_bwd, oracle_bwd
    x = _case(i)
    G = x["H"] // x["qk_heads"]
    gr = synth.make_bwd_inputs(x)
    io = x["q"].dtype
    state = x["h0"].dtype if x["h0"] is not None else torch.float32
    gr = {"do": gr["do"].float().to(io), "dv_in": gr["dv_in"].float().to(io), "dht": gr["dht"].to(state)}
    d, gd = to_dev(x), to_dev(gr)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda")
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
            workspace=ws, beta_logits=x["beta_logits"])
    gpu = kda.bwd_dh(x["scale"], gd["do"], gd["dv_in"], gd["dht"], dims, ws)
    torch.cuda.synchronize()
    xe = dict(x)
    xe["q"] = x["q"].repeat_interleave(G, dim=2)
    xe["k"] = x["k"].repeat_interleave(G, dim=2)
    if x["beta_logits"]:
        xe["beta"] = torch.sigmoid(x["beta"].double())
    res = compare_bwd(x, (gpu[0], gpu[1].float(), gpu[2].float()), oracle_bwd(xe, gr))
    assert_bwd_within(res, f"case {i}")
