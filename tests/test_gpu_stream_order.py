"""Stream order around a forward whose kernels are chained by programmatic
dependent launch: device work that writes the inputs right before kda.fwd,
and device work that reads o right after it, on the same stream and with no
synchronisation in between, must see the forward in its place.  The result
equals that of the same forward on inputs prepared beforehand, bit for bit."""
from __future__ import annotations

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import make, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("B,T,H,plan", [(2, 4096, 32, "two-stage"), (1, 4096, 16, "segmented"),
                                        (1, 8269, 32, "staged")])
def test_inputs_written_and_output_read_on_the_same_stream(B, T, H, plan):
    x = synth.make_inputs(make(B=B, T=T, H=H, seed=T + H))
    d = to_dev(x)
    # reference: inputs prepared and synchronised first
    v2 = (d["v"].float() * 2).to(torch.bfloat16)
    g2 = d["g"] * 0.5
    o_ref, ht_ref = kda.fwd(d["q"], d["k"], v2, g2, d["beta"], d["scale"], h0=d["h0"])
    torch.cuda.synchronize()
    # the same, with the inputs rewritten in place by device work right before
    # the call and o consumed by device work right after it
    v = d["v"].clone()
    g = d["g"].clone()
    torch.cuda.synchronize()
    for _ in range(3):
        v.copy_(d["v"])
        g.copy_(d["g"])
        v.mul_(2)
        g.mul_(0.5)
        o, ht = kda.fwd(d["q"], d["k"], v, g, d["beta"], d["scale"], h0=d["h0"])
        s = (o.float() * 1.0).sum()  # reads o on the same stream
        v.zero_()                    # and overwrites an input the forward has read
        g.zero_()
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(ht, ht_ref)
    assert torch.isclose(s, o_ref.float().sum())
    lay = kda.workspace_layout(kda.make_dims(B, T, H, 128, 128))
    got = "segmented" if lay.seg_count > 1 else "staged" if lay.stage_count > 1 else "two-stage"
    assert got == plan
