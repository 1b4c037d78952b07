"""GPU parity of the segmented scan (few sequences x heads over long
sequences): per-segment affine maps, their fp32 chaining, and the output pass
over all segments in parallel, against the fp64 oracle.  Each case first
checks that the workspace plan really cuts its sequences into segments."""
from __future__ import annotations

import pytest
import torch

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import synth
from parity_util import assert_within, compare, make, oracle_ref, run_gpu, to_dev

pytestmark = pytest.mark.gpu


def plan(x):
    d = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else x["N"])
    return kda.workspace_layout(d)


def full_check(x, what, min_segments=2):
    assert plan(x).seg_count >= min_segments, what
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    res = compare(x, o, ht, o_ref, ht_ref)
    assert_within(res, what)
    return o, ht


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64), (64, 128)])
def test_two_heads_ragged_tail(K, V):
    x = synth.make_inputs(make(B=1, T=64 * 100 + 17, H=2, K=K, V=V, seed=300 + K + V))
    full_check(x, f"segmented K{K} V{V}")


def test_many_short_segments_k64():
    x = synth.make_inputs(make(B=2, T=64 * 100 + 5, H=1, K=64, V=64, seed=311))
    assert plan(x).seg_count >= 2
    full_check(x, "six segments")


def test_varlen_uneven_segment_counts():
    """Sequences of different segment counts (and an empty one) in one pack, with h0."""
    lengths = [5000, 1, 0, 3000, 2048]
    x = synth.make_inputs(make(T=0, H=2, seed=321), lengths=lengths)
    x["h0"] = 0.1 * torch.randn((len(lengths), 2, 128, 128), generator=torch.Generator().manual_seed(5))
    o, ht = full_check(x, "varlen segmented")
    torch.testing.assert_close(ht[2].cpu(), x["h0"][2], rtol=0, atol=0)  # empty sequence


def test_segmented_with_variants():
    """fp16 I/O, bf16 state and grouped heads through the segmented path."""
    from test_gpu_variants import errors, oracle_variant, run_variant
    x = synth.make_variant_inputs(make(B=1, T=64 * 100 + 30, H=4, seed=331), io_dtype=torch.float16,
                                  qk_heads=2, state_dtype=torch.bfloat16)
    assert plan(x).seg_count >= 2
    o, ht = run_variant(x)
    o_ref, ht_ref = oracle_variant(x)
    assert_within(errors(x, o, ht, o_ref, ht_ref), "segmented variants")


def test_long_k64_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["long_k64"])
    assert plan(x).seg_count >= 2
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "long_k64")


def test_segmented_deterministic():
    x = synth.make_inputs(make(B=1, T=64 * 100 + 17, H=2, seed=341))
    a = run_gpu(x)
    b = run_gpu(x)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
