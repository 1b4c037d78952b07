"""The C-ABI calls are asynchronous and allocate nothing when the caller
passes the workspace, so a training or serving loop can capture them into a
CUDA graph and replay it.  Replays must reproduce the eager results bit for
bit, and pick up new input values written into the captured buffers."""
from __future__ import annotations

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import make, to_dev

pytestmark = pytest.mark.gpu


def _setup(x):
    d = to_dev(x)
    dims = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else x["N"])
    ws = kda.new_workspace(dims, "cuda")
    o = torch.empty((x["B"], x["T"], x["H"], x["V"]), dtype=torch.bfloat16, device="cuda")
    ht = torch.empty((x["N"], x["H"], x["K"], x["V"]), dtype=torch.float32, device="cuda")
    return d, dims, ws, o, ht


@pytest.mark.parametrize("lengths", [None, [300, 0, 64, 1000]])
def test_forward_graph_replay_matches_eager(lengths):
    x = synth.make_inputs(make(B=1 if lengths else 2, T=0 if lengths else 1000, H=4, seed=51), lengths=lengths)
    if lengths is None:
        x["h0"] = 0.1 * torch.randn((x["N"], 4, 128, 128), generator=torch.Generator().manual_seed(2))
    d, dims, ws, o, ht = _setup(x)

    def run(stream):
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                workspace=ws, out=o, final_state=ht, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(s)  # warm-up (loads the library, sets kernel attributes) outside the capture
    torch.cuda.synchronize()
    o_eager, ht_eager = o.clone(), ht.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    o.zero_()
    ht.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_eager) and torch.equal(ht, ht_eager)
    assert kda.status(ws) == 0

    # new values in the captured input buffers flow through the replay
    d["v"].mul_(2)
    if d["h0"] is not None:
        d["h0"].mul_(2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, 2 * o_eager)  # linear in (v, h0); power-of-two scaling is exact
    assert torch.equal(ht, 2 * ht_eager)


def test_backward_graph_replay_matches_eager():
    x = synth.make_inputs(make(B=2, T=700, H=2, seed=53))
    gr = {k_: (v_.cuda() if v_ is not None else None) for k_, v_ in synth.make_bwd_inputs(x).items()}
    d, dims, ws, o, ht = _setup(x)
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws, out=o, final_state=ht)
    lay = kda.workspace_layout(dims)
    dhck = torch.empty((lay.max_chunks, 2, 128, 128), dtype=torch.bfloat16, device="cuda")
    dv2 = torch.zeros((2, 700, 2, 128), dtype=torch.bfloat16, device="cuda")
    dh0 = torch.empty((2, 2, 128, 128), dtype=torch.float32, device="cuda")
    lib = kda.load_library()
    import ctypes
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731

    def run(stream):
        rc = lib.kda_bwd_dh(ctypes.c_float(x["scale"]), P(gr["do"]), P(gr["dv_in"]), P(gr["dht"]), P(dhck), P(dv2),
                            P(dh0), ctypes.byref(dims), P(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(s)
    torch.cuda.synchronize()
    ref = (dhck.clone(), dv2.clone(), dh0.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    dhck.zero_()
    dv2.zero_()
    dh0.zero_()
    g.replay()
    torch.cuda.synchronize()
    nchunks = 2 * ((700 + 63) // 64)
    assert torch.equal(dhck[:nchunks], ref[0][:nchunks])
    assert torch.equal(dv2, ref[1]) and torch.equal(dh0, ref[2])
