"""Parity of the intra-chunk stage's own outputs (the workspace: qg, kg, w, u,
Aqk, gd) against the fp64 chunked oracle, chunk by chunk, and of the scan at
the chunk counts where a two-deep ring first reuses its stages."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from oracle import chunked as oc
from parity_util import assert_within, compare, make, oracle_ref, run_gpu, to_dev

pytestmark = pytest.mark.gpu

REL = {"qg": 5e-3, "kg": 5e-3, "w": 5e-3, "u": 5e-3, "Aqk": 5e-3, "gd": 1e-6}
# Per (chunk, head) tile, so that one wrong tile is not diluted by the rest:
# relative error at twice the pooled bound (every element is one bf16 rounding
# of an fp32 result) and max|x - x_ref| <= 2e-2 * max|x_ref|, the element bound
# of the forward's output, on tiles of at least 16 valid rows (fewer elements
# make the relative error a small-sample statistic); gd (an fp32 sum of at
# most 64 terms in another order) to 1e-5 of the tile's largest |G|.
TILE_REL = 1e-2
TILE_MAXREL = 2e-2
TILE_MIN_ROWS = 16
GD_TILE_MAXREL = 1e-5


def _region(ws, off, count, dtype):
    nbytes = count * torch.tensor([], dtype=dtype).element_size()
    return ws[off:off + nbytes].view(dtype)


def _tile_check(name, got, want, where, worst):
    nb = np.linalg.norm(want)
    mb = np.max(np.abs(want)) if want.size else 0.0
    if nb == 0:
        assert np.all(got == 0), (name, where)
        return
    rel = np.linalg.norm(got - want) / nb
    mrel = np.max(np.abs(got - want)) / mb
    worst[name] = max(worst.get(name, 0.0), rel)
    assert rel <= TILE_REL, (name, where, rel)
    assert mrel <= TILE_MAXREL, (name, where, mrel)


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64)])
def test_workspace_intermediates_match_chunked_oracle(K, V):
    lengths = [130, 64, 1, 77, 1000]
    x = synth.make_inputs(make(T=0, H=2, K=K, V=V, seed=120 + K + V), lengths=lengths)
    d = to_dev(x)
    dims = kda.make_dims(1, x["T"], 2, K, V, len(lengths))
    ws = kda.new_workspace(dims, "cuda")
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
            workspace=ws)
    torch.cuda.synchronize()
    lay = kda.workspace_layout(dims)
    H, C = 2, 64
    tiles = lay.max_chunks * H
    wsc = ws.cpu()
    got = {
        "qg": _region(wsc, lay.qg, tiles * C * K, torch.bfloat16).view(lay.max_chunks, H, C, K),
        "kg": _region(wsc, lay.kg, tiles * C * K, torch.bfloat16).view(lay.max_chunks, H, C, K),
        "w": _region(wsc, lay.w, tiles * C * K, torch.bfloat16).view(lay.max_chunks, H, C, K),
        "u": _region(wsc, lay.u, tiles * C * V, torch.bfloat16).view(lay.max_chunks, H, C, V),
        "Aqk": _region(wsc, lay.aqk, tiles * C * C, torch.bfloat16).view(lay.max_chunks, H, C, C),
        "gd": _region(wsc, lay.gd, tiles * K, torch.float32).view(lay.max_chunks, H, K),
    }
    cu = np.concatenate([[0], np.cumsum(lengths)])
    f = lambda t: t.double().numpy()  # noqa: E731
    q, k, v, g, beta = (f(x[n])[0] for n in ("q", "k", "v", "g", "beta"))
    got_all = {n: [] for n in got}
    want_all = {n: [] for n in got}
    worst = {}
    base = 0
    for s, n in enumerate(lengths):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            chunks = oc.chunk_intra(q[a:b, h], k[a:b, h], v[a:b, h], g[a:b, h], beta[a:b, h], x["scale"], C)
            for c, ch in enumerate(chunks):
                t = base + c
                vr = ch["valid"]
                where = (s, c, h)
                for name in ("qg", "kg", "w", "u"):
                    gv = got[name][t, h].double().numpy()
                    got_all[name].append(gv[:vr].ravel())
                    want_all[name].append(ch[name][:vr].ravel())
                    assert np.all(gv[vr:] == 0), f"{name} padding rows of sequence {s} chunk {c} are not zero"
                    if vr >= TILE_MIN_ROWS:
                        _tile_check(name, gv[:vr], ch[name][:vr], where, worst)
                ga = got["Aqk"][t, h].double().numpy()
                got_all["Aqk"].append(ga[:vr, :vr].ravel())
                want_all["Aqk"].append(ch["Aqk"][:vr, :vr].ravel() / x["scale"])  # stored without scale
                assert np.all(np.triu(ga, 1) == 0), "Aqk above the diagonal is not zero"
                if vr >= TILE_MIN_ROWS:
                    _tile_check("Aqk", np.tril(ga[:vr, :vr]), np.tril(ch["Aqk"][:vr, :vr]) / x["scale"], where, worst)
                gg = got["gd"][t, h].double().numpy()
                got_all["gd"].append(gg)
                want_all["gd"].append(ch["G"])
                assert np.max(np.abs(gg - ch["G"])) <= GD_TILE_MAXREL * max(np.max(np.abs(ch["G"])), 1e-30), where
        base += len(chunks) if n > 0 else 0
    pooled = {}
    for name, tol in REL.items():
        a, b = np.concatenate(got_all[name]), np.concatenate(want_all[name])
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        pooled[name] = rel
        assert rel <= tol, (name, rel)
    print(f"[parity] intermediates K={K} V={V}: pooled " + " ".join(f"{n}={v:.2e}" for n, v in pooled.items())
          + "; worst tile " + " ".join(f"{n}={v:.2e}" for n, v in worst.items()), flush=True)


@pytest.mark.parametrize("nt", [2, 3, 5])
def test_ring_reuse_chunk_counts(nt):
    """Chunk counts 2, 3 and 5 (a two-stage ring's first reuse and beyond),
    forward and reverse scan, against the oracle."""
    from test_gpu_bwd import assert_bwd_within, compare_bwd, oracle_bwd, run_bwd
    x = synth.make_inputs(make(B=2, T=64 * nt - 3, H=2, seed=130 + nt))
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), f"NT {nt}")
    gr = synth.make_bwd_inputs(x)
    assert_bwd_within(compare_bwd(x, run_bwd(x, gr), oracle_bwd(x, gr)), f"bwd NT {nt}")
