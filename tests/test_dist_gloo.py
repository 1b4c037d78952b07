"""Multi-rank host logic on CPU (gloo, world_size 2): a batch is sharded into
contiguous blocks of (sequence, head) units, one per rank, with no exchange on
the data path; only the timing is reduced (max over ranks).  Each rank cuts
its block out of the batch with the same helpers the GPU path uses
(dist.plan_shard / take_shard: a batch slice, or a packed block with
cu_seqlens rebased to 0 and the matching h0 rows, or a block of heads), runs
the oracle on it as a problem of its own in place of the GPU kernel, and the
blocks, placed back with dist.place_shard, must reassemble to the single-rank
result bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from chunked_gated_delta_gb300 import dist as kdist


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CASES = {
    "packed": dict(lengths=[37, 0, 64, 130, 5], B=1, T=0, H=3),   # sequence blocks, rebased offsets
    "fixed": dict(lengths=None, B=3, T=70, H=3),                 # batch slices
    "heads": dict(lengths=None, B=1, T=90, H=5),                  # one sequence: blocks of heads
}


def _inputs(case):
    from chunked_gated_delta_gb300 import synth
    c = CASES[case]
    w = synth.Workload("dist", B=c["B"], T=c["T"], H=c["H"], K=16, V=8, seed=123)
    return synth.make_inputs(w, lengths=c["lengths"])


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = kdist.rank_info()
        assert (r, w, lr) == (rank, world, rank)
        for case in CASES:
            x = _inputs(case)
            cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].tolist()
            sh = kdist.plan_shard(x["B"], x["T"], x["H"], r, w, cu)
            q, k, v, g, beta, h0, lcu = kdist.take_shard(sh, x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                         x["h0"], x["cu_seqlens"])
            if lcu is not None:
                assert int(lcu[0]) == 0 and int(lcu[-1]) == q.shape[1]
            o, ht = oracle.recurrent_fwd(q, k, v, g, beta, x["scale"], h0=h0, cu_seqlens=lcu)
            np.save(os.path.join(out_dir, f"{case}_o{rank}.npy"), o)
            np.save(os.path.join(out_dir, f"{case}_ht{rank}.npy"), ht)
        assert kdist.max_over_ranks(float(rank + 1), w) == float(world)
        kdist.barrier(w)
    finally:
        dist.destroy_process_group()


def test_shard_range_tiles_exactly():
    for n in (0, 1, 5, 7, 128):
        for world in (1, 2, 3, 8):
            spans = [kdist.shard_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        kdist.shard_range(4, 2, 2)
    assert kdist.job_throughput([100, 300], 2.0) == 200.0


def test_plan_shard_covers_every_unit_once():
    for B, T, H, cu in [(4, 100, 3, None), (1, 100, 8, None), (1, 0, 4, [0, 5, 5, 9, 20, 20, 31])]:
        for world in (1, 2, 3, 5):
            seen = []
            for r in range(world):
                sh = kdist.plan_shard(B, T, H, r, world, cu)
                seen += [(s, h) for s in range(sh.s0, sh.s1) for h in range(sh.h0, sh.h1)]
                if cu is not None:
                    assert (sh.r0, sh.r1) == (cu[sh.s0], cu[sh.s1])
            N = B if cu is None else len(cu) - 1
            assert sorted(seen) == [(s, h) for s in range(N) for h in range(H)], (B, H, cu, world)


def test_two_rank_gloo_sharding(tmp_path):
    import oracle
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    for case in CASES:
        x = _inputs(case)
        o_full, ht_full = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                               h0=x["h0"], cu_seqlens=x["cu_seqlens"])
        o = np.full_like(o_full, np.nan)
        ht = np.full_like(ht_full, np.nan)
        cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].tolist()
        for r in range(world):
            sh = kdist.plan_shard(x["B"], x["T"], x["H"], r, world, cu)
            kdist.place_shard(sh, np.load(tmp_path / f"{case}_o{r}.npy"), np.load(tmp_path / f"{case}_ht{r}.npy"),
                              o, ht)
        np.testing.assert_array_equal(o, o_full)
        np.testing.assert_array_equal(ht, ht_full)


# ------------------------------------------------------------------ context parallel (T split)

def _cp_inputs():
    from chunked_gated_delta_gb300 import synth
    w = synth.Workload("cp", B=2, T=300, H=2, K=16, V=8, seed=321)
    return synth.make_inputs(w)


def _oracle_map(q, k, v, g, beta, scale):
    """[P | Q] of a token range by the oracle: P from h0 = I with v = 0 (the
    state map alone), Q from h0 = 0; fp64 [B, H, K, K + V]."""
    import torch

    import oracle
    B, T, H, K = q.shape
    eye = torch.eye(K, dtype=torch.float32).expand(B, H, K, K).contiguous()
    v0 = torch.zeros((B, T, H, K), dtype=torch.bfloat16)
    _, P = oracle.recurrent_fwd(q, k, v0, g, beta, scale, h0=eye)
    _, Q = oracle.recurrent_fwd(q, k, v, g, beta, scale, h0=None)
    return np.concatenate([P, Q], axis=-1)


def _cp_worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x = _cp_inputs()
        t0, t1 = kdist.plan_time_shard(x["T"], rank, world)
        loc = {n: x[n][:, t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")}
        pq = torch.from_numpy(_oracle_map(loc["q"], loc["k"], loc["v"], loc["g"], loc["beta"], x["scale"]))
        parts = [torch.empty_like(pq) for _ in range(world)]
        dist.all_gather(parts, pq)  # the one exchange, in rank order
        K = x["K"]
        h = x["h0"].double().numpy()
        for r in range(rank):  # the chain: h_in[r + 1] = P_r h_in[r] + Q_r
            P, Q = parts[r].numpy()[..., :K], parts[r].numpy()[..., K:]
            h = np.einsum("bhij,bhjv->bhiv", P, h) + Q
        f64 = {n: loc[n].double() for n in loc}  # the exact input values; the entry state stays fp64
        o, ht = oracle.recurrent_fwd(f64["q"], f64["k"], f64["v"], f64["g"], f64["beta"], x["scale"],
                                     h0=h, fp64_inputs=True)
        np.save(os.path.join(out_dir, f"cp_o{rank}.npy"), o)
        np.save(os.path.join(out_dir, f"cp_ht{rank}.npy"), ht)
        np.save(os.path.join(out_dir, f"cp_hin{rank}.npy"), h)
    finally:
        dist.destroy_process_group()


def test_plan_time_shard_covers_the_sequence():
    for T in (0, 1, 63, 64, 65, 300, 4097):
        for world in (1, 2, 3, 8):
            spans = [kdist.plan_time_shard(T, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            assert all(a[0] % 64 == 0 or a[0] == T for a in spans)  # chunk boundaries (or an empty tail)


def test_two_rank_gloo_context_parallel(tmp_path):
    """Two gloo ranks split two sequences of 300 tokens along T: each maps its
    range ([P | Q] by the oracle), the maps are all-gathered, each chains them
    into its entry state and runs its range from there.  The concatenated
    outputs and the last rank's final state equal the unsplit oracle to fp64
    rounding (the composition only reassociates the same products)."""
    import oracle
    world = 2
    mp.spawn(_cp_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    x = _cp_inputs()
    o_full, ht_full = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"])
    o = np.concatenate([np.load(tmp_path / f"cp_o{r}.npy") for r in range(world)], axis=1)
    ht = np.load(tmp_path / f"cp_ht{world - 1}.npy")
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)  # noqa: E731
    assert rel(o, o_full) < 1e-10 and rel(ht, ht_full) < 1e-10
    # rank 1's entry state is the state after rank 0's tokens
    t0, t1 = kdist.plan_time_shard(x["T"], 0, world)
    _, h_mid = oracle.recurrent_fwd(*(x[n][:, t0:t1].contiguous() for n in ("q", "k", "v", "g", "beta")),
                                    x["scale"], h0=x["h0"])
    assert rel(np.load(tmp_path / "cp_hin1.npy"), h_mid) < 1e-10
