"""The staged forward: one long sequence whose scan leaves most SMs idle runs
as chunk ranges, the intra-chunk kernel of range j + 1 beside the scan of
range j, with the fp32 state handed from range to range through the
workspace.

Checked against the fp64 oracle (the forward's tolerances), bit for bit
against the unstaged path (kda_fwd_intra then kda_fwd_scan, which take the
same arithmetic in the same order), through the interface variants, a packed
single sequence, CUDA graph capture, and the reverse state scan that reads
the staged forward's workspace.
"""
from __future__ import annotations

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from chunked_gated_delta_gb300.binding import IO_F16, STATE_BF16
from parity_util import assert_within, compare, make, oracle_ref, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def _dims(x):
    return kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else x["N"])


def _stages(x):
    L = kda.workspace_layout(_dims(x))
    return L.stage_count, L.stage_len


def _unstaged(x, ws=None):
    """kda_fwd_intra then kda_fwd_scan on one stream: the same kernels over every chunk at once."""
    d = to_dev(x)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda") if ws is None else ws
    o = torch.empty((x["B"], x["T"], x["H"], x["V"]), dtype=torch.bfloat16, device="cuda")
    ht = torch.empty((x["N"], x["H"], x["K"], x["V"]), dtype=torch.float32, device="cuda")
    kda.fwd_intra(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], dims, ws)
    kda.fwd_scan(d["scale"], d["h0"], o, ht, dims, ws)
    torch.cuda.synchronize()
    assert kda.status(ws) == 0
    return o, ht


# (T, H, K, V, expected stage count, stage length)
SHAPES = [
    (8192, 32, 128, 128, 2, 64),
    (8269, 32, 128, 128, 2, 65),     # ragged last chunk, uneven ranges
    (12293, 32, 128, 128, 3, 65),    # three ranges, the last one shorter
    (8192, 32, 64, 128, 2, 64),
    (8192, 64, 64, 64, 2, 64),
    (8192, 64, 128, 64, 2, 64),
]


@pytest.mark.parametrize("T,H,K,V,P,Lp", SHAPES)
def test_staged_matches_oracle_and_unstaged_bitwise(T, H, K, V, P, Lp):
    x = synth.make_inputs(make(B=1, T=T, H=H, K=K, V=V, seed=61 + T + H))
    assert _stages(x) == (P, Lp)
    o, ht = run_gpu(x)
    o_u, ht_u = _unstaged(x)
    assert torch.equal(o, o_u) and torch.equal(ht, ht_u)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), (T, H, K, V))


def test_staged_without_initial_or_final_state():
    x = synth.make_inputs(make(B=1, T=8269, H=32, h0=False, seed=71))
    assert _stages(x)[0] == 2
    o, ht = run_gpu(x, want_ht=False)
    assert ht is None
    o_u, _ = _unstaged(x)
    assert torch.equal(o, o_u)
    o_ref, _ = oracle_ref(x, want_ht=False)
    assert_within(compare(x, o, None, o_ref, None), "no h0, no ht")


def test_staged_packed_single_sequence():
    # cu_seqlens = [0, T]: the planner's tables, one sequence
    x = synth.make_inputs(make(B=1, T=0, H=32, seed=72), lengths=[9000])
    assert _stages(x)[0] == 2
    o, ht = run_gpu(x)
    o_u, ht_u = _unstaged(x)
    assert torch.equal(o, o_u) and torch.equal(ht, ht_u)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "packed single sequence")


def test_staged_interface_variants_bitwise():
    # fp16 I/O, bf16 state, beta logits and grouped value heads through the ranges
    w = make(B=1, T=8269, H=32, seed=73)
    x = synth.make_variant_inputs(w, io_dtype=torch.float16, qk_heads=8, beta_logits=True,
                                  state_dtype=torch.bfloat16)
    assert kda.workspace_layout(kda.make_dims(1, x["T"], 32, 128, 128)).stage_count == 2
    d = to_dev(x)
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], beta_logits=True)
    # the unstaged reference: the same call split into its two stages through the C ABI
    import ctypes
    lib = kda.load_library()
    dims = kda.make_dims(1, x["T"], 32, 128, 128)
    opts = kda.FwdOpts(IO_F16, STATE_BF16, 1, 8)
    ws = kda.new_workspace(dims, "cuda")
    o2 = torch.empty_like(o)
    ht2 = torch.empty_like(ht)
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.kda_fwd_intra_ex(P(d["q"]), P(d["k"]), P(d["v"]), P(d["g"]), P(d["beta"]), None,
                                ctypes.byref(dims), ctypes.byref(opts), P(ws), ctypes.c_size_t(ws.numel()), s) == 0
    assert lib.kda_fwd_scan_ex(ctypes.c_float(d["scale"]), P(d["h0"]), P(o2), P(ht2), ctypes.byref(dims),
                               ctypes.byref(opts), P(ws), ctypes.c_size_t(ws.numel()), s) == 0
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(ht, ht2)


def test_staged_graph_capture_replays_bitwise():
    x = synth.make_inputs(make(B=1, T=8269, H=32, seed=74))
    d = to_dev(x)
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda")
    o = torch.empty((1, x["T"], 32, 128), dtype=torch.bfloat16, device="cuda")
    ht = torch.empty((1, 32, 128, 128), dtype=torch.float32, device="cuda")

    def run(stream):
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws, out=o,
                final_state=ht, stream=stream)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run(s)  # the first staged call on the device creates the library's streams: outside the capture
    torch.cuda.synchronize()
    o_e, ht_e = o.clone(), ht.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    o.zero_()
    ht.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, o_e) and torch.equal(ht, ht_e)
    d["v"].mul_(2)
    d["h0"].mul_(2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, 2 * o_e) and torch.equal(ht, 2 * ht_e)
    assert kda.status(ws) == 0


def test_reverse_scan_reads_the_staged_workspace():
    x = synth.make_inputs(make(B=1, T=8269, H=32, seed=75))
    gr = synth.make_bwd_inputs(x)
    dims = _dims(x)
    d, gd = to_dev(x), to_dev(gr)
    outs = []
    for staged in (True, False):
        ws = kda.new_workspace(dims, "cuda")
        if staged:
            kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws)
        else:
            _unstaged(x, ws)
        outs.append(kda.bwd_dh(x["scale"], gd["do"], gd["dv_in"], gd["dht"], dims, ws))
        torch.cuda.synchronize()
        assert kda.status(ws) == 0
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_staged_back_to_back_calls_on_two_streams():
    # two staged forwards from different caller streams share the library's
    # streams; each must still see only its own inputs
    xs = [synth.make_inputs(make(B=1, T=8192, H=32, seed=80 + i)) for i in range(2)]
    refs = [_unstaged(x) for x in xs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    ds = [to_dev(x) for x in xs]
    torch.cuda.synchronize()
    outs = []
    for d, s in zip(ds, streams):
        with torch.cuda.stream(s):
            outs.append(kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], stream=s))
    torch.cuda.synchronize()
    for (o, ht), (o_u, ht_u) in zip(outs, refs):
        assert torch.equal(o, o_u) and torch.equal(ht, ht_u)
