"""The sharded forward on one GPU: every rank's block of a batch (dist.plan_shard:
blocks of whole sequences, or of heads for a single sequence) run through
the library one after the other, placed back with dist.place_shard, gives
the unsharded call's o and ht bit for bit.  The ranks here are sequential
host calls on one GPU (nothing waits on another rank), which is what each of
N GPUs would run on its own block."""
import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import dist as kdist
from chunked_gated_delta_gb300 import synth
from parity_util import make, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.mark.parametrize("case", ["fixed", "fixed_wide", "packed", "heads"])
@pytest.mark.parametrize("world", [2, 3])
def test_shards_reassemble_bitwise(case, world):
    if case == "fixed":
        x = synth.make_inputs(make(B=4, T=333, H=4, seed=141))
    elif case == "fixed_wide":   # 32 heads: the unsharded scan takes 128-column tiles, the shards 64-column ones
        x = synth.make_inputs(make(B=4, T=300, H=32, seed=142))
    elif case == "packed":
        x = synth.make_inputs(make(T=0, H=3, seed=143), lengths=[70, 1, 0, 300, 64, 129, 5])
        x["h0"] = 0.1 * torch.randn((7, 3, 128, 128), generator=torch.Generator().manual_seed(144))
    else:
        x = synth.make_inputs(make(B=1, T=700, H=6, seed=145))
    d = to_dev(x)
    o_full, ht_full = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                              cu_seqlens=d["cu_seqlens"])
    o = torch.full_like(o_full, float("nan"))
    ht = torch.full_like(ht_full, float("nan"))
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].tolist()
    for r in range(world):
        sh = kdist.plan_shard(x["B"], x["T"], x["H"], r, world, cu)
        o_l, ht_l = kdist.fwd_shard(sh, d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                                    cu_seqlens=d["cu_seqlens"])
        kdist.place_shard(sh, o_l, ht_l, o, ht)
    torch.cuda.synchronize()
    assert torch.equal(o, o_full)
    assert torch.equal(ht, ht_full)
