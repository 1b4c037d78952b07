"""Guard regions around every buffer the kernels write.

Each output (o, ht, dhck, dv2, dh0) and the workspace sit in the middle of a
larger allocation whose head and tail are filled with a byte pattern; after
the forward and the reverse scan the pattern must be intact, on the plain,
packed, segmented and staged paths.  A kernel that stores past the end of a
buffer (or before its start) changes a guard byte.  Outputs are also checked
against the unguarded calls bit for bit.
"""
from __future__ import annotations

import ctypes

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import make, to_dev

pytestmark = pytest.mark.gpu

GUARD = 1 << 16  # bytes before and after each buffer (a multiple of 256: alignment is kept)
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape`/`dtype` inside a pattern-filled byte allocation."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        return bool((self.raw[:GUARD] == PATTERN).all()) and bool((self.raw[GUARD + self.nbytes:] == PATTERN).all())


def _dims(x):
    return kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else x["N"])


CASES = {
    "plain": lambda: synth.make_inputs(make(B=2, T=300, H=3, seed=91)),
    "packed": lambda: synth.make_inputs(make(B=1, T=0, H=4, seed=92), lengths=[130, 0, 64, 1, 700]),
    "segmented": lambda: synth.make_inputs(make(B=1, T=4100, H=16, seed=93)),
    "staged": lambda: synth.make_inputs(make(B=1, T=8269, H=32, seed=94)),
}


@pytest.mark.parametrize("case", list(CASES))
def test_no_store_outside_any_buffer(case):
    x = CASES[case]()
    dims = _dims(x)
    lay = kda.workspace_layout(dims)
    if case == "segmented":
        assert lay.seg_count > 1
    if case == "staged":
        assert lay.stage_count > 1
    B, T, H, K, V, N = x["B"], x["T"], x["H"], x["K"], x["V"], x["N"]
    d = to_dev(x)
    ws = Guarded((kda.workspace_size(dims),), torch.uint8)
    o = Guarded((B, T, H, V), torch.bfloat16)
    ht = Guarded((N, H, K, V), torch.float32)
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
            workspace=ws.t, out=o.t, final_state=ht.t)
    torch.cuda.synchronize()
    assert kda.status(ws.t) == 0
    assert ws.intact() and o.intact() and ht.intact(), case
    o_ref, ht_ref = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                            cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    assert torch.equal(o.t, o_ref) and torch.equal(ht.t, ht_ref)

    # the reverse state scan on the same (guarded) workspace
    gr = to_dev(synth.make_bwd_inputs(x))
    dhck = Guarded((lay.max_chunks, H, K, V), torch.bfloat16)
    dv2 = Guarded((B, T, H, V), torch.bfloat16)
    dv2.t.zero_()  # rows no sequence owns are not written
    dh0 = Guarded((N, H, K, V), torch.float32)
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())  # noqa: E731
    rc = kda.load_library().kda_bwd_dh(ctypes.c_float(x["scale"]), P(gr["do"]), P(gr["dv_in"]), P(gr["dht"]),
                                       P(dhck.t), P(dv2.t), P(dh0.t), ctypes.byref(dims), P(ws.t),
                                       ctypes.c_size_t(ws.t.numel()),
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    assert kda.status(ws.t) == 0
    assert ws.intact() and dhck.intact() and dv2.intact() and dh0.intact(), case
    ck_ref, dv2_ref, dh0_ref = kda.bwd_dh(x["scale"], gr["do"], gr["dv_in"], gr["dht"], dims, ws.t)
    torch.cuda.synchronize()
    tiles = int(kda.workspace_layout(dims).max_chunks)
    if x["cu_seqlens"] is not None:  # checkpoint slots past the chunk table are unused
        cu = x["cu_seqlens"].tolist()
        tiles = sum((cu[i + 1] - cu[i] + 63) // 64 for i in range(len(cu) - 1))
    assert torch.equal(dhck.t[:tiles], ck_ref[:tiles]) and torch.equal(dv2.t, dv2_ref)
    assert torch.equal(dh0.t, dh0_ref)
