"""Multi-rank host logic on CPU (gloo, world_size 2): sharding of (sequence,
head) units across ranks needs no exchange on the data path; only the timing
is reduced (max over ranks).  Each rank runs the oracle on its shard in place
of the GPU kernel, and the shards must reassemble to the single-rank result."""
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


def _lengths():
    return [37, 0, 64, 130, 5]


def _inputs():
    from chunked_gated_delta_gb300 import synth
    w = synth.Workload("dist", B=1, T=0, H=3, K=16, V=8, seed=123)
    return synth.make_inputs(w, lengths=_lengths())


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist

    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = kdist.rank_info()
        assert (r, w, lr) == (rank, world, rank)
        x = _inputs()
        s0, s1 = kdist.shard_range(x["N"], r, w)
        units = [(s, h) for s in range(s0, s1) for h in range(x["H"])]
        o, ht = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"], h0=x["h0"],
                                     cu_seqlens=x["cu_seqlens"], units=units)
        np.save(os.path.join(out_dir, f"o{rank}.npy"), o)
        np.save(os.path.join(out_dir, f"ht{rank}.npy"), ht)
        np.save(os.path.join(out_dir, f"range{rank}.npy"), np.array([s0, s1]))
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


def test_two_rank_gloo_sharding(tmp_path):
    import oracle
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    x = _inputs()
    o_full, ht_full = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                           h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    cu = x["cu_seqlens"].tolist()
    covered = []
    for r in range(world):
        s0, s1 = np.load(tmp_path / f"range{r}.npy")
        o = np.load(tmp_path / f"o{r}.npy")
        ht = np.load(tmp_path / f"ht{r}.npy")
        for s in range(s0, s1):
            covered.append(s)
            np.testing.assert_array_equal(o[:, cu[s]:cu[s + 1]], o_full[:, cu[s]:cu[s + 1]])
            np.testing.assert_array_equal(ht[s], ht_full[s])
    assert sorted(covered) == list(range(x["N"]))
