"""The single-pass fused forward (kda_fwd_ex with KDA_PLAN_FUSED): every valid
element against the fp64 oracle on small ragged shapes, packed batches with
empty sequences, the exact gate path and the five named workloads.  The fused
kernel runs the intra-chunk stage and the scan step of each chunk with the
same arithmetic as the two kernels, so where the two-stage plan is neither
segmented nor different in its state hand-off it gives the same bits."""
import numpy as np
import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import assert_within, compare, make, oracle_ref, report, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def run(x, plan, want_ht=True, workspace=None):
    d = to_dev(x)
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                    output_final_state=want_ht, plan=plan, workspace=workspace)
    torch.cuda.synchronize()
    return o, ht


def _dims(x):
    return kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else x["N"])


def check(x, what, bitwise=None):
    """Fused against the oracle (every element) and against the two stages:
    bit for bit unless the two-stage plan segments the scan."""
    ws = kda.new_workspace(_dims(x), "cuda")
    o, ht = run(x, "fused", workspace=ws)
    assert kda.status(ws) == 0
    o_ref, ht_ref = oracle_ref(x)
    res = compare(x, o, ht, o_ref, ht_ref)
    report(f"fused {what}", res)
    assert_within(res, what)
    if bitwise is None:
        bitwise = kda.workspace_layout(_dims(x)).seg_count == 1
    o2, ht2 = run(x, "two_stage")
    if bitwise:
        assert torch.equal(o, o2) and torch.equal(ht, ht2), what
    return o, ht


@pytest.mark.parametrize("K,V", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_small_shapes_ragged(K, V, T):
    x = synth.make_inputs(make(B=2, T=T, H=3, K=K, V=V, seed=T * 11 + K + V))
    check(x, f"K={K} V={V} T={T}")


def test_no_initial_and_no_final_state():
    x = synth.make_inputs(make(B=1, T=300, H=2, h0=False, seed=201))
    check(x, "h0=None")
    x = synth.make_inputs(make(B=1, T=300, H=2, seed=202))
    o, ht = run(x, "fused", want_ht=False)
    assert ht is None
    o_ref, _ = oracle_ref(x, want_ht=False)
    assert_within(compare(x, o, None, o_ref, None), "ht not requested")


def test_packed_with_empty_and_edge_lengths():
    lengths = [1, 0, 63, 64, 65, 130, 0, 7]
    x = synth.make_inputs(make(T=0, H=3, seed=203), lengths=lengths)
    x["h0"] = 0.1 * torch.randn((len(lengths), 3, 128, 128), generator=torch.Generator().manual_seed(204))
    o, ht = check(x, "packed")
    for s, n in enumerate(lengths):
        if n == 0:
            torch.testing.assert_close(ht[s].cpu(), x["h0"][s], rtol=0, atol=0)


def test_strong_decay_takes_the_exact_path():
    x = synth.make_inputs(make(B=1, T=200, H=2, mu=-6.0, seed=205))
    dims = _dims(x)
    ws = kda.new_workspace(dims, "cuda")
    run(x, "fused", workspace=ws)
    assert kda.exact_path_tiles(ws, dims) > 0
    check(x, "strong decay")


def test_deterministic():
    x = synth.make_inputs(make(B=2, T=333, H=4, seed=206))
    a = run(x, "fused")
    b = run(x, "fused")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_interface_variants_are_unsupported():
    x = synth.make_variant_inputs(make(B=1, T=100, H=2, seed=207), io_dtype=torch.float16)
    d = to_dev(x)
    with pytest.raises(kda.KdaError) as e:
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], plan="fused")
    assert e.value.code == 2  # KDA_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["tiny", "mid", "headline", "varlen", "long"])
def test_named_workloads(name):
    x = synth.make_inputs(synth.WORKLOADS[name])
    check(x, name)
