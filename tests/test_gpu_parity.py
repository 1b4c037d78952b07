"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case compares every valid element of o and ht, the full-size workloads
included (in the launch configuration the benchmark times).  Tolerances are
those of the forward with bf16 I/O and fp32 accumulation (parity_util.REL_O /
MAXREL_O / REL_HT over the pooled elements, and UNIT_REL for each (sequence,
head) unit on its own).
"""
import numpy as np
import pytest
import torch

from chunked_gated_delta_gb300 import synth
from parity_util import assert_within, compare, make, oracle_ref, report, run_gpu, to_dev

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


def full_check(x, want_ht=True, what=""):
    o, ht = run_gpu(x, want_ht=want_ht)
    o_ref, ht_ref = oracle_ref(x, want_ht=want_ht)
    res = compare(x, o, ht, o_ref, ht_ref)
    report(what, res)
    assert_within(res, what)
    return res


# ------------------------------------------------------------------ small, every element

def test_tiny_workload():
    x = synth.make_inputs(synth.WORKLOADS["tiny"])
    full_check(x, what="tiny")


@pytest.mark.parametrize("K,V", [(128, 128), (64, 128), (128, 64), (64, 64)])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_small_shapes_ragged(K, V, T):
    x = synth.make_inputs(make(B=2, T=T, H=3, K=K, V=V, seed=T * 7 + K + V))
    full_check(x, what=f"K={K} V={V} T={T}")


@pytest.mark.parametrize("K,V,H", [(128, 128, 80), (64, 64, 80), (64, 128, 80)])
def test_many_heads_scan_variants(K, V, H):
    """Enough (sequence, head) units that the scan switches tile shape: a
    128-wide V tile per head (V = 128) or two 64-wide CTAs per SM (V = 64)."""
    x = synth.make_inputs(make(B=2, T=130, H=H, K=K, V=V, seed=H + K + V))
    full_check(x, what=f"many heads K={K} V={V}")


def test_no_initial_state_and_no_final_state():
    x = synth.make_inputs(make(B=1, T=300, H=2, h0=False, seed=5))
    full_check(x, what="h0=None")
    x = synth.make_inputs(make(B=1, T=300, H=2, seed=6))
    o, ht = run_gpu(x, want_ht=False)
    assert ht is None
    o_ref, _ = oracle_ref(x, want_ht=False)
    assert_within(compare(x, o, None, o_ref, None), "ht not requested")


def test_varlen_small_with_empty_and_edge_lengths():
    lengths = [1, 0, 63, 64, 65, 130, 0, 7]
    x = synth.make_inputs(make(T=0, H=3, seed=11), lengths=lengths)
    x["h0"] = 0.1 * torch.randn((len(lengths), 3, 128, 128), generator=torch.Generator().manual_seed(3))
    res = full_check(x, what="varlen small")
    o, ht = run_gpu(x)
    for s, L in enumerate(lengths):
        if L == 0:
            torch.testing.assert_close(ht[s].cpu(), x["h0"][s], rtol=0, atol=0)
    assert res


def test_strong_decay_takes_exact_path():
    """Decay so strong that gate factors would overflow: the exact per-element path."""
    x = synth.make_inputs(make(B=1, T=200, H=2, mu=-6.0, seed=21))
    full_check(x, what="strong decay")


def test_near_full_forget_invariant():
    """g = -80 (a finite stand-in for -inf) and beta = 1: o_t = scale (q_t . k_t) v_t."""
    x = synth.make_inputs(make(B=1, T=150, H=2, seed=31))
    x["g"] = torch.full_like(x["g"], -80.0)
    x["beta"] = torch.ones_like(x["beta"])
    o, ht = run_gpu(x)
    q, k, v = (x[n].double() for n in ("q", "k", "v"))
    want = x["scale"] * (q * k).sum(-1, keepdim=True) * v
    got = o.double().cpu()
    err = (got - want).norm() / want.norm()
    assert err < 5e-3, float(err)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "g=-80")


@pytest.mark.parametrize("K", [64, 128])
def test_beta0_g0_keeps_the_state(K):
    """beta = 0 and g = 0: nothing is written or forgotten, so ht = h0 exactly
    (the state update adds exact zeros) and o_t = scale * h0^T q_t, up to the
    bf16 copy of h0 the output product reads."""
    x = synth.make_inputs(make(B=2, T=333, H=3, K=K, V=K, seed=35))
    x["beta"] = torch.zeros_like(x["beta"])
    x["g"] = torch.zeros_like(x["g"])
    o, ht = run_gpu(x)
    assert torch.equal(ht.cpu(), x["h0"])
    want = x["scale"] * torch.einsum("bthk,bhkv->bthv", x["q"].double(), x["h0"].double())
    got = o.double().cpu()
    assert float((got - want).norm() / want.norm()) < 5e-3
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "beta=0, g=0")


@pytest.mark.parametrize("K", [64, 128])
def test_orthonormal_keys_recall(K):
    """beta = 1, g = 0, h0 = 0 and K orthonormal keys (one per token, T = K):
    the final state recalls every value, ht^T k_j = v_j, to the precision of
    the bf16 keys and intermediates; and the result matches the oracle."""
    T = K
    x = synth.make_inputs(make(B=1, T=T, H=2, K=K, V=K, h0=False, seed=36))
    gen = torch.Generator().manual_seed(37)
    keys = []
    for _ in range(2):
        Qm, _ = torch.linalg.qr(torch.randn((K, K), generator=gen, dtype=torch.float64))
        keys.append(Qm.T)  # rows orthonormal
    x["k"] = torch.stack(keys, dim=1).unsqueeze(0).to(torch.bfloat16)  # [1, T, 2, K]
    x["beta"] = torch.ones_like(x["beta"])
    x["g"] = torch.zeros_like(x["g"])
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "orthonormal recall")
    for h in range(2):
        kk = x["k"][0, :, h].double()                         # [T, K]
        recall = (ht[0, h].double().cpu().T @ kk.T).T           # [T, V]
        v = x["v"][0, :, h].double()
        assert float((recall - v).norm() / v.norm()) < 3e-2, h


# ------------------------------------------------------------------ named workloads

def test_mid_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["mid"])
    full_check(x, what="mid")


def test_varlen_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["varlen"])
    full_check(x, what="varlen")


def test_headline_workload_full():
    x = synth.make_inputs(synth.WORKLOADS["headline"])
    full_check(x, what="headline")


def test_long_workload_full():
    """One 65536-token sequence of 32 heads: the staged forward (chunk ranges
    of the intra kernel beside the scan), every element against the oracle."""
    x = synth.make_inputs(synth.WORKLOADS["long"])
    full_check(x, what="long")


# ------------------------------------------------------------------ metamorphic (bitwise)

def _small():
    return synth.make_inputs(make(B=2, T=190, H=3, seed=41))


def test_power_of_two_scaling_is_exact():
    x = _small()
    o1, h1 = run_gpu(x)
    y = dict(x, v=(x["v"].float() * 2).to(torch.bfloat16), h0=x["h0"] * 2)
    o2, h2 = run_gpu(y)
    assert torch.equal(o2.float(), 2 * o1.float())
    assert torch.equal(h2, 2 * h1)
    z = dict(x, scale=2 * x["scale"])
    o3, h3 = run_gpu(z)
    assert torch.equal(o3.float(), 2 * o1.float())
    assert torch.equal(h3, h1)


def test_head_and_batch_permutation_equivariance():
    x = _small()
    o1, h1 = run_gpu(x)
    perm = torch.tensor([2, 0, 1])
    y = dict(x)
    for n in ("q", "k", "v", "g"):
        y[n] = x[n][:, :, perm].contiguous()
    y["beta"] = x["beta"][:, :, perm].contiguous()
    y["h0"] = x["h0"][:, perm].contiguous()
    o2, h2 = run_gpu(y)
    assert torch.equal(o2, o1[:, :, perm])
    assert torch.equal(h2, h1[:, perm])
    bperm = torch.tensor([1, 0])
    z = dict(x)
    for n in ("q", "k", "v", "g", "beta"):
        z[n] = x[n][bperm].contiguous()
    z["h0"] = x["h0"][bperm].contiguous()
    o3, h3 = run_gpu(z)
    assert torch.equal(o3, o1[bperm])
    assert torch.equal(h3, h1[bperm])


def test_deterministic_and_workspace_contents_do_not_matter():
    import chunked_gated_delta_gb300 as kda
    x = _small()
    d = to_dev(x)
    dims = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"])
    ws = kda.new_workspace(dims, "cuda")
    ws.fill_(0xFF)  # NaN bit patterns everywhere
    o1, h1 = run_gpu(x, workspace=ws)
    ws.fill_(0x00)
    o2, h2 = run_gpu(x, workspace=ws)
    o3, h3 = run_gpu(x)
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    assert torch.equal(h1, h2) and torch.equal(h1, h3)
    assert kda.status(ws) == 0
    del d


def test_causal_bitwise():
    x = _small()
    o1, _ = run_gpu(x)
    t0 = 100  # inside the second chunk
    y = dict(x)
    gen = torch.Generator().manual_seed(9)
    for n in ("q", "k", "v"):
        t = x[n].clone()
        t[:, t0 + 1:] = torch.randn(t[:, t0 + 1:].shape, generator=gen).to(t.dtype)
        y[n] = t
    b = x["beta"].clone()
    b[:, t0 + 1:] = 0.5
    y["beta"] = b
    o2, _ = run_gpu(y)
    assert torch.equal(o1[:, :t0 + 1], o2[:, :t0 + 1])
    assert not torch.equal(o1[:, t0 + 1:], o2[:, t0 + 1:])


def test_varlen_writes_only_its_rows():
    import chunked_gated_delta_gb300 as kda
    lengths = [70, 1, 129]
    x = synth.make_inputs(make(T=0, H=2, seed=51), lengths=lengths)
    d = to_dev(x)
    T = sum(lengths)
    big = torch.full((1, T + 64, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    o = big[:, :T]
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
            cu_seqlens=d["cu_seqlens"], out=o)
    torch.cuda.synchronize()
    assert torch.all(big[:, T:] == 7.0)
    o_ref, _ = oracle_ref(x, want_ht=False)
    assert_within(compare(x, o, None, o_ref, None), "varlen canary")


def test_bad_seqlens_reported():
    import chunked_gated_delta_gb300 as kda
    x = synth.make_inputs(make(T=0, H=2, seed=61), lengths=[10, 20])
    d = to_dev(x)
    d["cu_seqlens"] = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")  # decreasing
    dims = kda.make_dims(1, 30, 2, 128, 128, num_seqs=2)
    ws = kda.new_workspace(dims, "cuda")
    o = torch.zeros((1, 30, 2, 128), dtype=torch.bfloat16, device="cuda")
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], cu_seqlens=d["cu_seqlens"],
            workspace=ws, out=o)
    assert kda.status(ws) == 7
    assert torch.all(o == 0)


def test_empty_batch_copies_h0():
    import chunked_gated_delta_gb300 as kda
    h0 = torch.randn((2, 3, 128, 128), device="cuda")
    z = torch.zeros((2, 0, 3, 128), dtype=torch.bfloat16, device="cuda")
    o, ht = kda.fwd(z, z, z, torch.zeros((2, 0, 3, 128), device="cuda"),
                    torch.zeros((2, 0, 3), dtype=torch.bfloat16, device="cuda"), 0.1, h0=h0)
    torch.cuda.synchronize()
    assert torch.equal(ht, h0)


def test_host_buffer_entry_point_matches_device_entry_point():
    """kda_fwd_host (host buffers, copies inside) gives the same bits as kda_fwd."""
    import chunked_gated_delta_gb300 as kda
    for x in (synth.make_inputs(make(B=2, T=130, H=2, seed=81)),
              synth.make_inputs(make(T=0, H=2, seed=82), lengths=[5, 70, 64])):
        o_dev, ht_dev = run_gpu(x)
        N = x["N"]
        dims = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"],
                             0 if x["cu_seqlens"] is None else N)
        arena = torch.empty(kda.host_arena_size(dims), dtype=torch.uint8, device="cuda")
        pin = {n: x[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
        h0 = x["h0"].pin_memory() if x["h0"] is not None else None
        cu = x["cu_seqlens"].pin_memory() if x["cu_seqlens"] is not None else None
        o = torch.empty((x["B"], x["T"], x["H"], x["V"]), dtype=torch.bfloat16, pin_memory=True)
        ht = torch.empty((N, x["H"], x["K"], x["V"]), dtype=torch.float32, pin_memory=True)
        kda.fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], x["scale"], h0, cu, o, ht,
                     dims, arena)
        torch.cuda.synchronize()
        assert torch.equal(o, o_dev.cpu())
        assert torch.equal(ht, ht_dev.cpu())


def test_bounded_wait_expires_and_context_survives():
    """A pipeline wait on a barrier nothing releases ends after its limit with
    KDA_ERR_TIMEOUT; the context then runs a normal forward correctly."""
    import time
    import chunked_gated_delta_gb300 as kda
    t0 = time.time()
    assert kda.selftest_wait_timeout(2_000_000) == 6  # 2 ms limit
    assert time.time() - t0 < 5.0
    x = synth.make_inputs(make(B=1, T=100, H=2, seed=91))
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "after timeout self-check")


@pytest.mark.parametrize("shape", ["fixed", "varlen"])
def test_host_entry_point_head_group_pipeline(shape):
    """Problems of 4096+ rows run kda_fwd_host as a pipeline, over time slices
    (fixed length) or head groups (packed): copies of one piece overlap the
    compute of the previous one.  The result matches the oracle and the
    device entry point (bit for bit for time slices: the same chunks, the
    state handed on in fp32)."""
    import chunked_gated_delta_gb300 as kda
    if shape == "fixed":
        x = synth.make_inputs(make(B=2, T=2100, H=8, seed=91))
        x["h0"] = 0.1 * torch.randn((2, 8, 128, 128), generator=torch.Generator().manual_seed(4))
    else:
        x = synth.make_inputs(make(T=0, H=4, seed=92), lengths=[3000, 0, 1500, 77])
    N = x["N"]
    dims = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"], 0 if x["cu_seqlens"] is None else N)
    arena = torch.empty(kda.host_arena_size(dims), dtype=torch.uint8, device="cuda")
    pin = {n: x[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    h0 = x["h0"].pin_memory() if x["h0"] is not None else None
    cu = x["cu_seqlens"].pin_memory() if x["cu_seqlens"] is not None else None
    o = torch.empty((x["B"], x["T"], x["H"], x["V"]), dtype=torch.bfloat16, pin_memory=True)
    ht = torch.empty((N, x["H"], x["K"], x["V"]), dtype=torch.float32, pin_memory=True)
    kda.fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], x["scale"], h0, cu, o, ht, dims, arena)
    torch.cuda.synchronize()
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), f"host pipeline {shape}")
    o_dev, ht_dev = run_gpu(x)
    torch.testing.assert_close(o.float(), o_dev.cpu().float(), rtol=2e-2, atol=2e-3)
    torch.testing.assert_close(ht, ht_dev.cpu(), rtol=1e-2, atol=1e-3)
    if shape == "fixed":
        assert torch.equal(o, o_dev.cpu()) and torch.equal(ht, ht_dev.cpu())


def _host_call(x, want_ht=True):
    import chunked_gated_delta_gb300 as kda
    dims = kda.make_dims(x["B"], x["T"], x["H"], x["K"], x["V"])
    arena = torch.empty(kda.host_arena_size(dims), dtype=torch.uint8, device="cuda")
    pin = {n: x[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    h0 = x["h0"].pin_memory() if x["h0"] is not None else None
    o = torch.empty((x["B"], x["T"], x["H"], x["V"]), dtype=torch.bfloat16, pin_memory=True)
    ht = torch.empty((x["B"], x["H"], x["K"], x["V"]), dtype=torch.float32, pin_memory=True) if want_ht else None
    kda.fwd_host(pin["q"], pin["k"], pin["v"], pin["g"], pin["beta"], x["scale"], h0, None, o, ht, dims, arena)
    torch.cuda.synchronize()
    return o, ht


def test_host_time_slices_ragged_bitwise():
    """Three sequences of 1537 tokens (a ragged last slice and chunk): kda_fwd_host
    over time slices gives the bits of kda_fwd, with and without ht."""
    x = synth.make_inputs(make(B=3, T=1537, H=32, seed=93))
    o, ht = _host_call(x)
    o_dev, ht_dev = run_gpu(x)
    assert torch.equal(o, o_dev.cpu()) and torch.equal(ht, ht_dev.cpu())
    o2, _ = _host_call(x, want_ht=False)
    assert torch.equal(o2, o)


def test_host_time_slices_long_sequence_bitwise():
    """One 65536-token sequence of 32 heads (each slice itself staged on the
    device; host rows of q, k, v, g, o of 512 MiB or more take one copy per
    sequence): the bits of
    kda_fwd."""
    x = synth.make_inputs(synth.WORKLOADS["long"])
    o, ht = _host_call(x)
    o_dev, ht_dev = run_gpu(x)
    assert torch.equal(o, o_dev.cpu()) and torch.equal(ht, ht_dev.cpu())


def test_varlen_thousands_of_short_sequences():
    """3000 packed sequences of 0-20 tokens (plus a few long ones): the
    planner's per-thread sequence ranges (more sequences than its threads),
    one-chunk sequences everywhere, and empty ones keeping h0."""
    rng = np.random.default_rng(77)
    lengths = [int(v) for v in rng.integers(0, 21, size=3000)]
    lengths[5] = 700
    lengths[2999] = 129
    x = synth.make_inputs(make(T=0, H=2, seed=97), lengths=lengths)
    x["h0"] = 0.1 * torch.randn((len(lengths), 2, 128, 128), generator=torch.Generator().manual_seed(6))
    o, ht = run_gpu(x)
    o_ref, ht_ref = oracle_ref(x)
    assert_within(compare(x, o, ht, o_ref, ht_ref), "3000 sequences")
    for s, n in enumerate(lengths):
        if n == 0:
            torch.testing.assert_close(ht[s].cpu(), x["h0"][s], rtol=0, atol=0)


# ------------------------------------------------------------------ both gate paths in one launch

def _exact_tiles_expected(x):
    """(chunk, head) tiles whose in-chunk log2 decay span exceeds 96 anywhere
    (the intra kernel's switch to exact per-element gates), from the inputs in
    fp64; the test inputs keep every tile far from the threshold."""
    g = x["g"].double().numpy()
    H = x["H"]
    cu = x["cu_seqlens"].tolist() if x["cu_seqlens"] is not None else None
    seqs = [(0, cu[s], cu[s + 1]) for s in range(len(cu) - 1)] if cu else [(b, 0, x["T"]) for b in range(x["B"])]
    exact, spans = set(), []
    for si, (b, a, e) in enumerate(seqs):
        for c0 in range(a, e, 64):
            blk = g[b, c0:min(c0 + 64, e)]                       # [rows, H, K]
            span = np.max(np.abs(np.cumsum(blk, axis=0) / np.log(2.0)), axis=(0, 2))  # per head
            for h in range(H):
                spans.append(span[h])
                if span[h] > 96.0:
                    exact.add((si, (c0 - a) // 64, h))
    spans = np.array(spans)
    assert np.all((spans < 48.0) | (spans > 192.0)), "a tile lies near the switch"
    return exact


def test_exact_and_factored_gate_paths_in_one_launch():
    """One launch whose tiles take both gate paths: sequence 0 has ordinary
    decay except for one chunk of very strong decay (whose gate factors would
    overflow: the exact per-element path), sequence 1 strong decay throughout,
    sequence 2 ordinary decay.  The kernel's count of exact-path tiles equals
    the count from the inputs, and each group of units matches the oracle."""
    import chunked_gated_delta_gb300 as kda
    lengths = [300, 200, 257]
    x = synth.make_inputs(make(T=0, H=4, seed=131), lengths=lengths)
    gen = torch.Generator().manual_seed(132)
    g = x["g"].clone()
    def strong(n):  # about -20 per token: even the 8-row tail chunk spans ~230 in log2
        return torch.nn.functional.logsigmoid(torch.randn((1, n) + tuple(g.shape[2:]), generator=gen) - 20.0)
    g[:, 64:128] = strong(64)                                    # sequence 0, chunk 1, every head
    g[:, 300:500] = strong(200)                                  # sequence 1, every chunk
    x["g"] = g
    want = _exact_tiles_expected(x)
    assert {c for (s, c, h) in want if s == 0} == {1} and len(want) == 4 + 4 * 4
    d = to_dev(x)
    dims = kda.make_dims(1, x["T"], 4, 128, 128, len(lengths))
    ws = kda.new_workspace(dims, "cuda")
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"],
                    cu_seqlens=d["cu_seqlens"], workspace=ws)
    assert kda.exact_path_tiles(ws, dims) == len(want)
    o_ref, ht_ref = oracle_ref(x)
    for name, units in (("mixed", [(0, h) for h in range(4)]), ("exact", [(1, h) for h in range(4)]),
                        ("factored", [(2, h) for h in range(4)])):
        res = compare(x, o, ht, o_ref, ht_ref, units)
        report(f"gate paths: {name}", res)
        assert_within(res, name)
    # an ordinary launch counts no exact-path tile
    y = synth.make_inputs(make(B=1, T=300, H=4, seed=133))
    dy = to_dev(y)
    dims_y = kda.make_dims(1, 300, 4, 128, 128)
    ws_y = kda.new_workspace(dims_y, "cuda")
    kda.fwd(dy["q"], dy["k"], dy["v"], dy["g"], dy["beta"], dy["scale"], h0=dy["h0"], workspace=ws_y)
    assert kda.exact_path_tiles(ws_y, dims_y) == 0 and not _exact_tiles_expected(y)


# ------------------------------------------------------------------ error budget

def test_error_budget_of_the_two_stages():
    """Where the forward's error comes from, on the mid workload: the fp64
    chunked scan run over the GPU's own bf16 intermediates (from the
    workspace) separates the intra stage's roundings (those intermediates
    against the exact ones) from the scan kernel's (its bf16 copies of h and
    v', fp32 accumulation, the final rounding of o).  Printed for the record;
    the asserts only bound each part by the forward's tolerance."""
    import chunked_gated_delta_gb300 as kda
    from oracle import chunked as oc
    x = synth.make_inputs(synth.WORKLOADS["mid"])
    d = to_dev(x)
    H, K, V, T, C = x["H"], x["K"], x["V"], x["T"], 64
    dims = kda.make_dims(1, T, H, K, V)
    ws = kda.new_workspace(dims, "cuda")
    o, ht = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], h0=d["h0"], workspace=ws)
    torch.cuda.synchronize()
    lay = kda.workspace_layout(dims)
    nc = lay.max_chunks
    wsc = ws.cpu()

    def region(off, count, dt, shape):
        n = count * torch.tensor([], dtype=dt).element_size()
        return wsc[off:off + n].view(dt).view(shape).double().numpy()

    qg = region(lay.qg, nc * H * C * K, torch.bfloat16, (nc, H, C, K))
    kg = region(lay.kg, nc * H * C * K, torch.bfloat16, (nc, H, C, K))
    w = region(lay.w, nc * H * C * K, torch.bfloat16, (nc, H, C, K))
    u = region(lay.u, nc * H * C * V, torch.bfloat16, (nc, H, C, V))
    aqk = region(lay.aqk, nc * H * C * C, torch.bfloat16, (nc, H, C, C))
    gd = region(lay.gd, nc * H * K, torch.float32, (nc, H, K))
    o_ref, ht_ref = oracle_ref(x)
    o_mid = np.zeros_like(o_ref)
    for h in range(H):
        chunks = [dict(qg=qg[c, h], kg=kg[c, h], w=w[c, h], u=u[c, h], Aqk=x["scale"] * aqk[c, h], G=gd[c, h],
                       valid=min(C, T - c * C)) for c in range((T + C - 1) // C)]
        o_mid[0, :, h], _ = oc.chunk_scan(chunks, x["h0"][0, h].double().numpy(), x["scale"])
    og = o.double().cpu().numpy()
    rel = lambda a, b: float(np.linalg.norm(a - b) / np.linalg.norm(b))  # noqa: E731
    total = rel(og, o_ref)
    intra = rel(o_mid, o_ref)          # the intermediates' roundings, scanned exactly
    scan = rel(og, o_mid)              # the scan kernel on those intermediates
    rounding = rel(torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy(), o_ref)  # o -> bf16 alone
    print(f"[budget] mid: total {total:.3e}; intra intermediates {intra:.3e}; scan kernel {scan:.3e} "
          f"(of which the bf16 rounding of o {rounding:.3e}); quadrature sum "
          f"{(intra ** 2 + scan ** 2) ** 0.5:.3e}", flush=True)
    assert total <= 5e-3 and intra <= 5e-3 and scan <= 5e-3
