"""Shared helpers of the GPU parity tests (comparison against the fp64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from chunked_gated_delta_gb300 import synth

# Tolerances of the forward: bf16 I/O with fp32 accumulation and state.
REL_O = 5e-3      # ||o - o_ref|| / ||o_ref||
MAXREL_O = 2e-2   # max|o - o_ref| <= MAXREL_O * max|o_ref|
REL_HT = 5e-3     # ||ht - ht_ref|| / ||ht_ref||


def to_dev(x, device="cuda"):
    out = {}
    for k_, v_ in x.items():
        out[k_] = v_.to(device) if isinstance(v_, torch.Tensor) else v_
    return out


def run_gpu(x, want_ht=True, workspace=None):
    import chunked_gated_delta_gb300 as kda
    d = to_dev(x)
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                    cu_seqlens=d["cu_seqlens"], output_final_state=want_ht, workspace=workspace)
    torch.cuda.synchronize()
    return o, ht


def oracle_ref(x, units=None, want_ht=True):
    return oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                cu_seqlens=x["cu_seqlens"], units=units, want_ht=want_ht)


def unit_rows(x, s, h):
    """Packed (batch, token) index arrays of sequence s: returns (b, t_slice)."""
    if x["cu_seqlens"] is None:
        return s, slice(0, x["T"])
    cu = x["cu_seqlens"].tolist()
    return 0, slice(cu[s], cu[s + 1])


def compare(x, o_gpu, ht_gpu, o_ref, ht_ref, units=None):
    """Error metrics over the valid elements of the selected units (fp64)."""
    o_g = o_gpu.float().cpu().numpy().astype(np.float64)
    H = x["H"]
    if units is None:
        units = [(s, h) for s in range(x["N"]) for h in range(H)]
    got, want = [], []
    for s, h in units:
        b, ts = unit_rows(x, s, h)
        got.append(o_g[b, ts, h].ravel())
        want.append(o_ref[b, ts, h].ravel())
    got = np.concatenate(got) if got else np.zeros(0)
    want = np.concatenate(want) if want else np.zeros(0)
    res = {}
    if want.size:
        assert np.all(np.isfinite(got)), "non-finite values in o"
        nref = np.linalg.norm(want)
        res["rel_o"] = float(np.linalg.norm(got - want) / max(nref, 1e-300))
        res["maxrel_o"] = float(np.max(np.abs(got - want)) / max(np.max(np.abs(want)), 1e-300))
    if ht_gpu is not None and ht_ref is not None:
        hg = ht_gpu.cpu().numpy().astype(np.float64)
        a = np.stack([hg[s, h] for s, h in units]) if units else np.zeros(0)
        r = np.stack([ht_ref[s, h] for s, h in units]) if units else np.zeros(0)
        if r.size and np.linalg.norm(r) > 0:
            assert np.all(np.isfinite(a)), "non-finite values in ht"
            res["rel_ht"] = float(np.linalg.norm(a - r) / np.linalg.norm(r))
        elif r.size:
            res["abs_ht"] = float(np.max(np.abs(a - r)))
    return res


def assert_within(res, what=""):
    if "rel_o" in res:
        assert res["rel_o"] <= REL_O, (what, res)
        assert res["maxrel_o"] <= MAXREL_O, (what, res)
    if "rel_ht" in res:
        assert res["rel_ht"] <= REL_HT, (what, res)
    if "abs_ht" in res:
        assert res["abs_ht"] <= 1e-6, (what, res)


def sample_units(x, n, seed=0, include=()):
    rng = np.random.default_rng(seed)
    all_units = [(s, h) for s in range(x["N"]) for h in range(x["H"])]
    idx = rng.choice(len(all_units), size=min(n, len(all_units)), replace=False)
    chosen = {all_units[i] for i in idx} | set(include)
    return sorted(chosen)


def make(name=None, **over):
    """Inputs of a named workload, or of an ad-hoc one built from keyword fields."""
    if name is not None:
        w = synth.WORKLOADS[name]
        if over:
            w = synth.Workload(**{**w.__dict__, **over})
    else:
        base = dict(name="adhoc", B=1, T=128, H=2, K=128, V=128, seed=99)
        base.update(over)
        w = synth.Workload(**base)
    return w
