"""GPU parity of the reverse state scan (kda_bwd_dh) against the fp64 oracle.

The GPU reads qg, kg, w and the chunk decay from the workspace of a forward
call on the same inputs (bf16 operands, fp32 state), the oracle recomputes
them in fp64 from the same bf16 inputs.  Tolerances are the forward's: every
operand of the three products per chunk is rounded to bf16 once (relative
error 2^-9) and accumulated in fp32, and dv2 is returned in bf16.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_gb300 import synth
from oracle import chunked as oc
from parity_util import UNIT_MIN_TOKENS, UNIT_REL, _Acc, make, to_dev

pytestmark = pytest.mark.gpu

REL = 5e-3      # ||x - x_ref|| / ||x_ref|| for dhck, dv2 and dh0
MAXREL = 2e-2   # max|x - x_ref| <= MAXREL * max|x_ref|


def _dims(x):
    import chunked_gated_delta_gb300 as kda
    return kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"],
                         0 if x["cu_seqlens"] is None else x["N"])


def run_bwd(x, gr, want_dhck=True, want_dh0=True, workspace=None):
    """Forward (to fill the workspace), then the reverse state scan."""
    import chunked_gated_delta_gb300 as kda
    d, gd = to_dev(x), to_dev(gr)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda") if workspace is None else workspace
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
            cu_seqlens=d["cu_seqlens"], output_final_state=False, workspace=ws)
    out = kda.bwd_dh(x["scale"], gd["do"], gd["dv_in"], gd["dht"], dims, ws,
                     want_dhck=want_dhck, want_dh0=want_dh0)
    torch.cuda.synchronize()
    assert kda.status(ws) == 0
    return out


def oracle_bwd(x, gr, units=None):
    f = lambda t: None if t is None else t.double().numpy()  # noqa: E731
    return oc.chunked_bwd_dh(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), x["scale"],
                             f(gr["do"]), f(gr["dv_in"]), dht=f(gr["dht"]),
                             cu_seqlens=None if x["cu_seqlens"] is None else x["cu_seqlens"].numpy(),
                             units=units)


def _bounds(x):
    if x["cu_seqlens"] is None:
        lens = [x["T"]] * x["B"]
        starts = [b * x["T"] for b in range(x["B"])]
    else:
        cu = x["cu_seqlens"].tolist()
        lens = [cu[s + 1] - cu[s] for s in range(len(cu) - 1)]
        starts = cu[:-1]
    tiles = [(n + 63) // 64 for n in lens]
    base = np.concatenate([[0], np.cumsum(tiles)]).astype(int)
    return starts, lens, base


def _metrics(got, want, what):
    got, want = np.concatenate(got), np.concatenate(want)
    if want.size == 0:
        return {}
    assert np.all(np.isfinite(got)), f"non-finite values in {what}"
    nref = np.linalg.norm(want)
    if nref == 0:
        return {f"abs_{what}": float(np.max(np.abs(got)))}
    return {f"rel_{what}": float(np.linalg.norm(got - want) / nref),
            f"maxrel_{what}": float(np.max(np.abs(got - want)) / np.max(np.abs(want)))}


def compare_bwd(x, gpu, ref, units=None):
    dhck_g, dv2_g, dh0_g = gpu
    dhck_r, dv2_r, dh0_r = ref
    H = x["H"]
    units = units or [(s, h) for s in range(x["N"]) for h in range(H)]
    starts, lens, base = _bounds(x)
    dv2_flat_g = dv2_g.float().cpu().numpy().astype(np.float64).reshape(-1, H, x["V"])
    dv2_flat_r = dv2_r.reshape(-1, H, x["V"])
    res = {}
    a, b = [], []
    for s, h in units:
        sl = slice(starts[s], starts[s] + lens[s])
        a.append(dv2_flat_g[sl, h].ravel())
        b.append(dv2_flat_r[sl, h].ravel())
    res.update(_metrics(a, b, "dv2"))
    if dhck_g is not None:
        ck = dhck_g[: int(base[-1])].float().cpu().numpy().astype(np.float64)  # slots past the table are unused
        a = [ck[base[s]:base[s + 1], h].ravel() for s, h in units]
        b = [dhck_r[base[s]:base[s + 1], h].ravel() for s, h in units]
        res.update(_metrics(a, b, "dhck"))
    if dh0_g is not None:
        d0 = dh0_g.cpu().numpy().astype(np.float64)
        res.update(_metrics([d0[s, h].ravel() for s, h in units], [dh0_r[s, h].ravel() for s, h in units],
                            "dh0"))
    return res


def assert_bwd_within(res, what=""):
    assert res, what
    for key, val in res.items():
        if key.startswith("rel_"):
            assert val <= REL, (what, res)
        elif key.startswith("maxrel_"):
            assert val <= MAXREL, (what, res)
        elif key.startswith("unit_"):
            assert val <= UNIT_REL, (what, res)
        else:
            assert val <= 1e-6, (what, res)


def full_bwd_check(x, gr, what="", **kw):
    gpu = run_bwd(x, gr, **kw)
    res = compare_bwd(x, gpu, oracle_bwd(x, gr))
    assert_bwd_within(res, what)
    return res


# ------------------------------------------------------------------ shapes

def test_tiny_workload():
    x = synth.make_inputs(synth.WORKLOADS["tiny"])
    full_bwd_check(x, synth.make_bwd_inputs(x), "tiny")


@pytest.mark.parametrize("K", [64, 128])
@pytest.mark.parametrize("V", [64, 128])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_small_shapes_ragged(K, V, T):
    x = synth.make_inputs(make(B=2, T=T, H=2, K=K, V=V, seed=5 + T + K + V))
    full_bwd_check(x, synth.make_bwd_inputs(x, seed=T), f"K{K} V{V} T{T}")


@pytest.mark.parametrize("K,V,H", [(128, 128, 96), (64, 64, 96), (64, 128, 96), (128, 64, 40)])
def test_many_heads_kernel_variants(K, V, H):
    """Enough (sequence, head, V tile) units to select the two-V-block and the
    single-stage kernels as well as the small-grid one."""
    x = synth.make_inputs(make(B=2, T=130, H=H, K=K, V=V, seed=H + V))
    full_bwd_check(x, synth.make_bwd_inputs(x), f"K{K} V{V} H{H}")


def test_no_dht_and_optional_outputs():
    x = synth.make_inputs(make(B=2, T=129, H=2, seed=41))
    gr = synth.make_bwd_inputs(x, dht=False)
    full_bwd_check(x, gr, "dht None")
    _, dv2_a, _ = run_bwd(x, gr)
    dhck, dv2_b, dh0 = run_bwd(x, gr, want_dhck=False, want_dh0=False)
    assert dhck is None and dh0 is None
    assert torch.equal(dv2_a, dv2_b)


def test_varlen_small_with_empty_and_edge_lengths():
    lengths = [1, 0, 63, 64, 65, 130, 0, 7]
    x = synth.make_inputs(make(T=0, H=3, seed=12), lengths=lengths)
    gr = synth.make_bwd_inputs(x)
    full_bwd_check(x, gr, "varlen small")
    _, _, dh0 = run_bwd(x, gr)
    for s, n in enumerate(lengths):
        if n == 0:  # no chunk: the gradient passes through unchanged
            torch.testing.assert_close(dh0[s].cpu(), gr["dht"][s], rtol=0, atol=0)


def test_strong_decay():
    x = synth.make_inputs(make(B=1, T=200, H=2, mu=-6.0, seed=22))
    full_bwd_check(x, synth.make_bwd_inputs(x), "strong decay")


def test_mid_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["mid"])
    full_bwd_check(x, synth.make_bwd_inputs(x), "mid")


# ------------------------------------------------------------------ full sizes, every element

def pooled_bwd_check(x, gr, gpu, what):
    """Every unit of a full-size workload against the fp64 oracle, run in a
    spawn process pool (tests/bwd_pool.py) and compared unit by unit as the
    results arrive (pooled norms plus each unit's own relative error)."""
    import bwd_pool
    dhck_g, dv2_g, dh0_g = gpu
    H, V = x["H"], x["V"]
    rows = x["B"] * x["T"]
    xn = {n: x[n].float().numpy().reshape((rows, H) + tuple(x[n].shape[3:])) for n in ("q", "k", "v", "g", "beta")}
    gn = {"do": gr["do"].float().numpy().reshape(rows, H, V), "dv_in": gr["dv_in"].float().numpy().reshape(rows, H, V),
          "dht": None if gr["dht"] is None else gr["dht"].float().numpy()}
    starts, lens, base = _bounds(x)
    dv2_n = dv2_g.float().cpu().numpy().reshape(rows, H, V)
    dhck_c = dhck_g.cpu()
    dh0_n = dh0_g.float().cpu().numpy()
    acc = {"dv2": _Acc(), "dhck": _Acc(), "dh0": _Acc()}
    units = [(s, h) for s in range(x["N"]) for h in range(H)]
    for (s, h), ck, d2, d0 in bwd_pool.map_units(bwd_pool.unit_jobs(xn, gn, x["scale"], units, starts, lens)):
        full = lens[s] >= UNIT_MIN_TOKENS
        acc["dv2"].add(dv2_n[starts[s]:starts[s] + lens[s], h], d2, (s, h), full)
        acc["dhck"].add(dhck_c[int(base[s]):int(base[s + 1]), h].double().numpy(), ck, (s, h), full)
        acc["dh0"].add(dh0_n[s, h], d0, (s, h), full)
    res = {}
    for name, a in acc.items():
        assert a.finite, f"non-finite values in {name}"
        if a.n and a.sr > 0:
            res[f"rel_{name}"] = a.rel()
            res[f"maxrel_{name}"] = a.maxrel()
            res[f"unit_{name}"] = a.worst
    print(f"[parity] bwd {what}: " + " ".join(f"{k}={v:.3e}" for k, v in res.items()), flush=True)
    assert_bwd_within(res, what)
    return res


def _full(name):
    x = synth.make_inputs(synth.WORKLOADS[name])
    gr = synth.make_bwd_inputs(x)
    gpu = run_bwd(x, gr)
    pooled_bwd_check(x, gr, gpu, name)
    return x, gr, gpu


def test_headline_workload_full_and_linear():
    x, gr, (dhck, dv2, dh0) = _full("headline")
    # the reverse scan is linear in (do, dv_in, dht): doubling them doubles every
    # output bit for bit (power-of-two scaling commutes with every rounding)
    gr2 = {k_: 2 * v_ for k_, v_ in gr.items()}
    dhck2, dv22, dh02 = run_bwd(x, gr2)
    assert torch.equal(dhck2, 2 * dhck)
    assert torch.equal(dv22, 2 * dv2)
    assert torch.equal(dh02, 2 * dh0)


def test_varlen_workload_full():
    _full("varlen")


def test_long_workload_full():
    _full("long")


def test_deterministic():
    x = synth.make_inputs(make(B=2, T=300, H=4, seed=8))
    gr = synth.make_bwd_inputs(x)
    a = run_bwd(x, gr)
    b = run_bwd(x, gr)
    for u, w in zip(a, b):
        assert torch.equal(u, w)


# ------------------------------------------------------------------ segmented reverse scan

def _seg_plan(x):
    import chunked_gated_delta_gb300 as kda
    return kda.workspace_layout(_dims(x))


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_segmented_two_heads_ragged(K, V):
    """Long sequence, few heads: maps of the newer segments, chained from dht,
    then every segment in parallel."""
    x = synth.make_inputs(make(B=1, T=64 * 100 + 17, H=2, K=K, V=V, seed=400 + K + V))
    assert _seg_plan(x).seg_count >= 2
    full_bwd_check(x, synth.make_bwd_inputs(x, seed=3), f"segmented K{K} V{V}")


def test_segmented_varlen_uneven_and_empty():
    lengths = [5000, 1, 0, 3000, 2048]
    x = synth.make_inputs(make(T=0, H=2, seed=411), lengths=lengths)
    assert _seg_plan(x).seg_count >= 2
    gr = synth.make_bwd_inputs(x)
    full_bwd_check(x, gr, "segmented varlen")
    _, _, dh0 = run_bwd(x, gr)
    torch.testing.assert_close(dh0[2].cpu(), gr["dht"][2], rtol=0, atol=0)  # empty sequence


def test_segmented_no_dht():
    x = synth.make_inputs(make(B=2, T=64 * 100 + 5, H=1, K=64, V=64, seed=421))
    assert _seg_plan(x).seg_count >= 2
    full_bwd_check(x, synth.make_bwd_inputs(x, dht=False), "segmented, dht None")


def test_long_k64_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["long_k64"])
    assert _seg_plan(x).seg_count >= 2
    gr = synth.make_bwd_inputs(x)
    pooled_bwd_check(x, gr, run_bwd(x, gr), "long_k64")


def test_grouped_value_heads():
    """The reverse scan runs per value head on the forward's workspace, so
    grouped q/k heads need nothing of it: compare with q/k expanded per value
    head in the oracle."""
    import chunked_gated_delta_gb300 as kda
    x = synth.make_variant_inputs(make(B=1, T=300, H=4, seed=431), qk_heads=2)
    gr = synth.make_bwd_inputs(x)
    d, gd = to_dev(x), to_dev(gr)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda")
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws)
    gpu = kda.bwd_dh(x["scale"], gd["do"], gd["dv_in"], gd["dht"], dims, ws)
    torch.cuda.synchronize()
    xe = dict(x)
    xe["q"] = x["q"].repeat_interleave(2, dim=2)
    xe["k"] = x["k"].repeat_interleave(2, dim=2)
    res = compare_bwd(x, gpu, oracle_bwd(xe, gr))
    assert_bwd_within(res, "grouped heads")



# ------------------------------------------------------------------ interface variants

@pytest.mark.parametrize("io,state", [(torch.float16, torch.float32), (torch.bfloat16, torch.bfloat16),
                                      (torch.float16, torch.bfloat16)])
@pytest.mark.parametrize("T", [130, 64 * 100 + 17])
def test_f16_gradients_and_bf16_state(io, state, T):
    """fp16 do / dv_in / dv2 and bf16 dht / dh0 (also through the segmented
    path at the longer length), against the oracle on the exact input values."""
    import chunked_gated_delta_gb300 as kda
    x = synth.make_inputs(make(B=1, T=T, H=2, seed=440 + T))
    gr = synth.make_bwd_inputs(x)
    gr = {"do": gr["do"].float().to(io), "dv_in": gr["dv_in"].float().to(io), "dht": gr["dht"].to(state)}
    d, gd = to_dev(x), to_dev(gr)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda")
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws)
    dhck, dv2, dh0 = kda.bwd_dh(x["scale"], gd["do"], gd["dv_in"], gd["dht"], dims, ws)
    torch.cuda.synchronize()
    assert dv2.dtype == io and dh0.dtype == state
    res = compare_bwd(x, (dhck, dv2.float(), dh0.float()), oracle_bwd(x, gr))
    assert_bwd_within(res, f"io {io} state {state} T {T}")
