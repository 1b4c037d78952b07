"""GPU parity of the forward's interface variants (kda_fwd_ex) against the
fp64 oracle: fp16 I/O, bf16 state I/O, beta given as logits (sigmoid on chip)
and grouped value heads (q / k shared by a group of value heads).

The oracle takes every variant through its plain definition: the exact input
values widened to fp64, q / k of value head h taken from q / k head
h // (H // Hqk), and beta = sigmoid(logit) computed in fp64.  Tolerances are
those of the default interface.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from chunked_gated_delta_gb300 import synth
from parity_util import REL_HT, assert_within, compare, make, to_dev

pytestmark = pytest.mark.gpu


def oracle_variant(x, units=None):
    G = x["H"] // x["qk_heads"]
    f64 = lambda t: t.double()  # noqa: E731
    q = f64(x["q"]).repeat_interleave(G, dim=2)
    k = f64(x["k"]).repeat_interleave(G, dim=2)
    beta = torch.sigmoid(f64(x["beta"])) if x["beta_logits"] else f64(x["beta"])
    h0 = None if x["h0"] is None else f64(x["h0"])
    return oracle.recurrent_fwd(q, k, f64(x["v"]), f64(x["g"]), beta, x["scale"], h0=h0,
                                cu_seqlens=x["cu_seqlens"], units=units, fp64_inputs=True)


def run_variant(x, want_ht=True):
    import chunked_gated_delta_gb300 as kda
    d = to_dev(x)
    state = x["h0"].dtype if x["h0"] is not None else x.get("state_dtype", torch.float32)
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                    cu_seqlens=d["cu_seqlens"], output_final_state=want_ht,
                    beta_logits=x["beta_logits"], state_dtype=state)
    torch.cuda.synchronize()
    return o, ht


def errors(x, o, ht, o_ref, ht_ref, units=None):
    return compare(x, o, ht, o_ref, ht_ref, units)


def check(x, what, units=None):
    o, ht = run_variant(x)
    o_ref, ht_ref = oracle_variant(x, units=units)
    res = errors(x, o, ht, o_ref, ht_ref, units)
    assert_within(res, what)
    return o, ht, res


# ------------------------------------------------------------------ fp16 I/O

@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (64, 128), (128, 64)])
@pytest.mark.parametrize("T", [1, 65, 200])
def test_f16_io_small(K, V, T):
    x = synth.make_variant_inputs(make(B=2, T=T, H=2, K=K, V=V, seed=T + K), io_dtype=torch.float16)
    o, ht, _ = check(x, f"f16 K{K} V{V} T{T}")
    assert o.dtype == torch.float16 and ht.dtype == torch.float32


def test_f16_io_strong_decay_exact_path():
    x = synth.make_variant_inputs(make(B=1, T=200, H=2, mu=-6.0, seed=23), io_dtype=torch.float16)
    check(x, "f16 strong decay")


def test_f16_io_mid_workload():
    x = synth.make_variant_inputs(synth.WORKLOADS["mid"], io_dtype=torch.float16)
    check(x, "f16 mid")


# ------------------------------------------------------------------ bf16 state I/O

def test_bf16_state_small_and_varlen():
    x = synth.make_variant_inputs(make(B=2, T=150, H=3, seed=61), state_dtype=torch.bfloat16)
    o, ht, _ = check(x, "bf16 state")
    assert ht.dtype == torch.bfloat16
    lengths = [5, 0, 64, 129, 1]
    x = synth.make_variant_inputs(make(T=0, H=2, seed=62), state_dtype=torch.bfloat16, lengths=lengths)
    o, ht, _ = check(x, "bf16 state varlen")
    # an empty sequence returns h0 unchanged (bf16 -> fp32 -> bf16 is exact)
    assert torch.equal(ht[1].cpu(), x["h0"][1])


def test_bf16_state_no_h0():
    x = synth.make_variant_inputs(make(B=1, T=100, H=2, seed=63, h0=False))
    x["state_dtype"] = torch.bfloat16
    o, ht = run_variant(x)
    assert ht.dtype == torch.bfloat16
    o_ref, ht_ref = oracle_variant(x)
    assert_within(errors(x, o, ht, o_ref, ht_ref), "bf16 state, no h0")


# ------------------------------------------------------------------ beta logits

@pytest.mark.parametrize("io", [torch.bfloat16, torch.float16])
def test_beta_logits(io):
    x = synth.make_variant_inputs(make(B=2, T=190, H=2, seed=71), io_dtype=io, beta_logits=True)
    check(x, f"beta logits {io}")


def test_beta_logits_matches_presigmoided_beta():
    """The in-kernel sigmoid agrees with applying it on the host first (to the
    bf16 rounding that separates the two beta inputs)."""
    import chunked_gated_delta_gb300 as kda
    x = synth.make_variant_inputs(make(B=1, T=128, H=2, seed=72), beta_logits=True)
    d = to_dev(x)
    o1, h1 = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], beta_logits=True)
    b2 = torch.sigmoid(d["beta"].float()).to(torch.bfloat16)
    o2, h2 = kda.fwd(d["q"], d["k"], d["v"], d["g"], b2, d["scale"], h0=d["h0"])
    err = (o1.float() - o2.float()).norm() / o2.float().norm()
    assert err < 5e-3, float(err)


# ------------------------------------------------------------------ grouped value heads

@pytest.mark.parametrize("H,Hqk", [(4, 1), (4, 2), (6, 3), (8, 8)])
def test_grouped_heads_small(H, Hqk):
    x = synth.make_variant_inputs(make(B=2, T=130, H=H, seed=80 + H + Hqk), qk_heads=Hqk)
    check(x, f"grouped H{H} Hqk{Hqk}")


def test_grouped_heads_equal_expanded_qk():
    """Grouped heads give exactly the result of q / k expanded to every value
    head (same kernels, same arithmetic per value head)."""
    import chunked_gated_delta_gb300 as kda
    x = synth.make_variant_inputs(make(B=1, T=200, H=4, seed=91), qk_heads=2)
    d = to_dev(x)
    o1, h1 = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"])
    qe, ke = (d[n].repeat_interleave(2, dim=2).contiguous() for n in ("q", "k"))
    o2, h2 = kda.fwd(qe, ke, d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"])
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_grouped_heads_headline_full():
    """Headline-sized grouped case (B=4, T=8192, 32 value heads over 8 q/k heads)."""
    x = synth.make_variant_inputs(synth.WORKLOADS["headline"], qk_heads=8)
    check(x, "grouped headline")


# ------------------------------------------------------------------ everything together

def test_all_variants_varlen():
    lengths = [70, 1, 0, 300, 64]
    x = synth.make_variant_inputs(make(T=0, H=4, seed=99), io_dtype=torch.float16, qk_heads=2,
                                  beta_logits=True, state_dtype=torch.bfloat16, lengths=lengths)
    o, ht, res = check(x, "all variants varlen")
    assert o.dtype == torch.float16 and ht.dtype == torch.bfloat16
    assert res["rel_ht"] <= REL_HT


def test_invalid_options_rejected():
    import chunked_gated_delta_gb300 as kda
    x = synth.make_variant_inputs(make(B=1, T=64, H=3, seed=7), qk_heads=3)
    d = to_dev(x)
    q2 = torch.zeros((1, 64, 2, 128), dtype=torch.bfloat16, device="cuda")  # 3 value heads over 2 q/k heads
    with pytest.raises(kda.KdaError):
        kda.fwd(q2, q2, d["v"], d["g"], d["beta"], d["scale"])
