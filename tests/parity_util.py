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


# A defect confined to a few heads or tiles is diluted in the pooled norms
# above, so every (sequence, head) unit with at least one full chunk is also
# held to its own relative error.  The bound is twice the pooled tolerance:
# a broken unit shows errors of order one, while a correct one sits at the
# pooled level (the same roundings over 64 x V or more elements).
UNIT_REL = 1e-2
UNIT_MIN_TOKENS = 64


class _Acc:
    """Streaming sums of one compared tensor (fp64): squared error and
    reference norms, maxima, and the worst per-unit relative error."""

    def __init__(self):
        self.se = self.sr = 0.0
        self.md = self.mr = 0.0
        self.worst = 0.0
        self.worst_unit = None
        self.n = 0
        self.finite = True

    def add(self, got, want, unit, weigh_unit=True):
        got = np.asarray(got, np.float64).ravel()
        want = np.asarray(want, np.float64).ravel()
        if want.size == 0:
            return
        self.finite &= bool(np.all(np.isfinite(got)))
        d = got - want
        se, sr = float(d @ d), float(want @ want)
        self.se += se
        self.sr += sr
        self.md = max(self.md, float(np.max(np.abs(d))))
        self.mr = max(self.mr, float(np.max(np.abs(want))))
        self.n += want.size
        if weigh_unit and sr > 0:
            r = (se / sr) ** 0.5
            if r > self.worst:
                self.worst, self.worst_unit = r, unit

    def rel(self):
        return (self.se / self.sr) ** 0.5 if self.sr > 0 else None

    def maxrel(self):
        return self.md / self.mr if self.mr > 0 else None


def compare(x, o_gpu, ht_gpu, o_ref, ht_ref, units=None):
    """Error metrics over the valid elements of the selected units (fp64),
    accumulated one (sequence, head) unit at a time."""
    o_g = o_gpu.float().cpu().numpy()  # exact for bf16 / fp16
    H = x["H"]
    if units is None:
        units = [(s, h) for s in range(x["N"]) for h in range(H)]
    ao, ah = _Acc(), _Acc()
    hg = ht_gpu.float().cpu().numpy() if (ht_gpu is not None and ht_ref is not None) else None
    abs_ht = 0.0
    for s, h in units:
        b, ts = unit_rows(x, s, h)
        n_tok = ts.stop - ts.start
        ao.add(o_g[b, ts, h], o_ref[b, ts, h], (s, h), n_tok >= UNIT_MIN_TOKENS)
        if hg is not None:
            ah.add(hg[s, h], ht_ref[s, h], (s, h), n_tok >= UNIT_MIN_TOKENS)
    res = {}
    if ao.n:
        assert ao.finite, "non-finite values in o"
        res["rel_o"] = ao.rel() if ao.rel() is not None else 0.0
        res["maxrel_o"] = ao.maxrel() if ao.maxrel() is not None else 0.0
        res["unit_rel_o"] = ao.worst
        res["unit_rel_o_at"] = ao.worst_unit
    if hg is not None and ah.n:
        assert ah.finite, "non-finite values in ht"
        if ah.sr > 0:
            res["rel_ht"] = ah.rel()
            res["unit_rel_ht"] = ah.worst
            res["unit_rel_ht_at"] = ah.worst_unit
        else:
            res["abs_ht"] = ah.md
    return res


def assert_within(res, what=""):
    if "rel_o" in res:
        assert res["rel_o"] <= REL_O, (what, res)
        assert res["maxrel_o"] <= MAXREL_O, (what, res)
        assert res["unit_rel_o"] <= UNIT_REL, (what, res)
    if "rel_ht" in res:
        assert res["rel_ht"] <= REL_HT, (what, res)
        assert res["unit_rel_ht"] <= UNIT_REL, (what, res)
    if "abs_ht" in res:
        assert res["abs_ht"] <= 1e-6, (what, res)


def report(what, res):
    """One line of parity figures on stdout (pytest -s shows it)."""
    keys = ("rel_o", "maxrel_o", "unit_rel_o", "rel_ht", "unit_rel_ht")
    figs = " ".join(f"{k}={res[k]:.3e}" for k in keys if k in res and res[k] is not None)
    print(f"[parity] {what}: {figs}", flush=True)


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
