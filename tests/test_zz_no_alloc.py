"""kda_fwd_noalloc: the forward for callers that cannot allocate device memory
(a plugin inside a framework whose allocator owns the GPU, or a
latency-critical path where cudaMalloc would synchronise the device).  Its
workspace is the library's built-in scratch array.

The test calls it through the C ABI on several problems in a row (two small
ones, then one long single sequence near the scratch capacity that takes the
segmented scan) and checks each result against kda_fwd with a
caller-allocated workspace and against the fp64 oracle, within the
tolerances of the parity tests.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import MAXREL_O, REL_HT, REL_O, assert_within, compare, make, oracle_ref, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    n = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / n), float(np.max(np.abs(a - b)) / np.max(np.abs(b)))


def _both(x):
    d = to_dev(x)
    o_ref, ht_ref = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                            cu_seqlens=d["cu_seqlens"])
    o = torch.full_like(o_ref, float("nan"))
    ht = torch.full_like(ht_ref, float("nan"))
    kda.fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["h0"], d["cu_seqlens"],
                    o, ht)
    torch.cuda.synchronize()
    return o, ht, o_ref, ht_ref


def test_noalloc_matches_kda_fwd_and_the_oracle_on_calls_in_a_row():
    first = synth.make_inputs(make(B=2, T=300, H=4, seed=71))
    second = synth.make_inputs(make(T=0, H=3, seed=72), lengths=[65, 1, 200, 64])
    # near the capacity at H = 1 (T <= 53248): one sequence whose scan is segmented
    third = synth.make_inputs(make(B=1, T=50000, H=1, seed=73))
    dims = kda.make_dims(1, 50000, 1, 128, 128)
    assert kda.workspace_layout(dims).seg_count > 1
    assert kda.workspace_size(dims) <= kda.binding.NOALLOC_SCRATCH_BYTES
    for x in (first, second, third):
        o, ht, o_dev, ht_dev = _both(x)
        rel, maxrel = _rel(o, o_dev)
        assert rel <= REL_O and maxrel <= MAXREL_O, (rel, maxrel)
        rel_h, _ = _rel(ht, ht_dev)
        assert rel_h <= REL_HT, rel_h
        o_ref, ht_ref = oracle_ref(x)
        assert_within(compare(x, o, ht, o_ref, ht_ref), "noalloc against the oracle")


def test_noalloc_rejects_problems_beyond_its_scratch():
    assert kda.workspace_size(kda.make_dims(1, 4096, 32, 128, 128)) > kda.binding.NOALLOC_SCRATCH_BYTES
    z = torch.zeros((1, 4096, 32, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((1, 4096, 32, 128), dtype=torch.float32, device="cuda")
    b = torch.zeros((1, 4096, 32), dtype=torch.bfloat16, device="cuda")
    ht = torch.zeros((1, 32, 128, 128), dtype=torch.float32, device="cuda")
    with pytest.raises(kda.KdaError) as e:
        kda.fwd_noalloc(z, z, z, g, b, 0.1, None, None, z, ht)
    assert e.value.code == 4  # KDA_ERR_WORKSPACE
