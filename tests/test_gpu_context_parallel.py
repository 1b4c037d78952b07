"""Context-parallel forward on one GPU: sequences split along T into ranges
(dist.plan_time_shard), each range's affine state map [P | Q] from
kda_fwd_state_map, the maps chained into entry states by kda_chain_states,
and each range finished by the scan from its entry state.  The ranks are
emulated as sequential host calls on one GPU (the exchange is a stack of the
maps); every element of the assembled o and the final state is compared with
the fp64 oracle of the unsplit sequences, and the maps themselves with the
oracle's (P from h0 = I with v = 0, Q from h0 = 0).  The tolerances are the
forward's: P and Q are computed with the bf16 operand copies the scan uses."""
import numpy as np
import pytest
import torch

import chunked_gated_delta_gb300 as kda
import oracle
from chunked_gated_delta_gb300 import dist as kdist
from chunked_gated_delta_gb300 import synth
from parity_util import REL_HT, assert_within, compare, make, oracle_ref, report, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

NAMES = ("q", "k", "v", "g", "beta")


def _oracle_map(x):
    """[P | Q] of the whole (packed or fixed) problem x, fp64 [N, H, K, K + V]."""
    B, T, H, K = x["q"].shape
    N = x["N"]
    eye = torch.eye(K, dtype=torch.float32).expand(N, H, K, K).contiguous()
    v0 = torch.zeros((B, T, H, K), dtype=torch.bfloat16)
    _, P = oracle.recurrent_fwd(x["q"], x["k"], v0, x["g"], x["beta"], x["scale"], h0=eye,
                                cu_seqlens=x["cu_seqlens"])
    _, Q = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=None,
                                cu_seqlens=x["cu_seqlens"])
    return np.concatenate([P, Q], axis=-1)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _p_bound(T):
    """P is the product of the range's chunk maps, each applied to a bf16 copy
    of the running product (relative rounding up to 2^-9 per chunk), so its
    relative error may grow linearly with the chunk count; Q is a state (from
    h0 = 0) and takes the forward's state tolerance."""
    return ((T + 63) // 64) * 2.0 ** -9


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64)])
@pytest.mark.parametrize("T", [130, 777])
def test_state_map_matches_the_oracle(K, V, T):
    x = synth.make_inputs(make(B=2, T=T, H=3, K=K, V=V, seed=151 + K + V + T))
    d = to_dev(x)
    pq, ws, dims = kda.state_map(d["q"], d["k"], d["v"], d["g"], d["beta"])
    torch.cuda.synchronize()
    assert kda.status(ws) == 0
    want = _oracle_map(x)
    got = pq.double().cpu().numpy()
    rp, rq = _rel(got[..., :K], want[..., :K]), _rel(got[..., K:], want[..., K:])
    print(f"[parity] state map K={K} V={V} T={T}: rel_P={rp:.3e} (bound {_p_bound(T):.2e}) rel_Q={rq:.3e}", flush=True)
    assert rp <= _p_bound(T), "P"
    assert rq <= REL_HT, "Q"


def test_state_map_of_empty_and_packed_sequences():
    lengths = [70, 0, 200, 1]
    x = synth.make_inputs(make(T=0, H=2, seed=161), lengths=lengths)
    d = to_dev(x)
    pq, _, _ = kda.state_map(d["q"], d["k"], d["v"], d["g"], d["beta"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    got = pq.double().cpu().numpy()
    K = x["K"]
    assert np.array_equal(got[1, :, :, :K], np.broadcast_to(np.eye(K), got[1, :, :, :K].shape))  # P = I
    assert np.all(got[1, :, :, K:] == 0)                                                         # Q = 0
    want = _oracle_map(x)
    for s in (0, 2, 3):
        assert _rel(got[s][..., :K], want[s][..., :K]) <= _p_bound(lengths[s]), s
        assert _rel(got[s][..., K:], want[s][..., K:]) <= REL_HT, s


@pytest.mark.parametrize("world", [2, 3, 5])
@pytest.mark.parametrize("K,V,h0", [(128, 128, True), (64, 64, False)])
def test_time_split_matches_the_oracle(world, K, V, h0):
    """Two sequences of 4113 tokens (a ragged end) split along T into `world`
    ranges; the assembled o and the last range's final state against the
    fp64 oracle of the whole sequences, and against the single-call forward."""
    x = synth.make_inputs(make(B=2, T=4113, H=3, K=K, V=V, h0=h0, seed=171 + world + K))
    d = to_dev(x)
    T = x["T"]
    maps, parts = [], []
    for r in range(world):
        t0, t1 = kdist.plan_time_shard(T, r, world)
        loc = {n: d[n][:, t0:t1].contiguous() for n in NAMES}
        pq, ws, dims = kdist.context_parallel_maps(*(loc[n] for n in NAMES))
        maps.append(pq)
        parts.append((t0, t1, ws, dims))
    pq_all = torch.stack(maps)  # the exchange, in rank order
    o = torch.full((x["B"], T, x["H"], V), float("nan"), dtype=torch.bfloat16, device="cuda")
    ht = None
    for r, (t0, t1, ws, dims) in enumerate(parts):
        o_r, ht_r = kdist.context_parallel_finish(pq_all, r, ws, dims, x["scale"], h0=d["h0"])
        o[:, t0:t1] = o_r
        ht = ht_r
        assert kda.status(ws) == 0
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle_ref(x)
    res = compare(x, o, ht, o_ref, ht_ref)
    report(f"time split world={world} K={K}", res)
    assert_within(res, f"time split {world}")
    o1, h1 = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"])
    assert _rel(o.double().cpu().numpy(), o1.double().cpu().numpy()) < 5e-3
    assert _rel(ht.double().cpu().numpy(), h1.double().cpu().numpy()) < 5e-3


def test_time_split_of_packed_sequences():
    """Packed sequences (one empty) with each sequence's tokens split into two
    ranges: every rank's local problem lists the same sequences (some empty)."""
    lengths = [300, 5, 0, 200]
    x = synth.make_inputs(make(T=0, H=2, seed=181), lengths=lengths)
    x["h0"] = 0.1 * torch.randn((4, 2, 128, 128), generator=torch.Generator().manual_seed(182))
    d = to_dev(x)
    cu = x["cu_seqlens"].tolist()
    world = 2
    maps, parts = [], []
    for r in range(world):
        spans = [kdist.plan_time_shard(n, r, world) for n in lengths]
        rows = [list(range(cu[s] + a, cu[s] + b)) for s, (a, b) in enumerate(spans)]
        idx = torch.tensor(sum(rows, []), dtype=torch.long, device="cuda")
        loc = {n: d[n][:, idx].contiguous() for n in NAMES}
        lcu = synth.cu_from_lengths([b - a for a, b in spans]).cuda()
        pq, ws, dims = kdist.context_parallel_maps(*(loc[n] for n in NAMES), cu_seqlens=lcu)
        maps.append(pq)
        parts.append((idx, ws, dims))
    pq_all = torch.stack(maps)
    o = torch.full((1, x["T"], 2, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    for r, (idx, ws, dims) in enumerate(parts):
        o_r, ht = kdist.context_parallel_finish(pq_all, r, ws, dims, x["scale"], h0=d["h0"])
        o[:, idx] = o_r
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle_ref(x)
    res = compare(x, o, ht, o_ref, ht_ref)
    assert_within(res, "packed time split")
    torch.testing.assert_close(ht[2].cpu(), x["h0"][2], rtol=0, atol=0)  # the empty sequence keeps h0
