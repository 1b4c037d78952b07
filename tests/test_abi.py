"""CPU checks of the C ABI: the library loads, exports every symbol the header
declares, sizes its workspace as documented, plans chunks as the pages' worked
examples do, and rejects bad arguments before touching a GPU."""
import ctypes
import json
import os
import re

import pytest

import chunked_gated_delta_gb300 as kda
from chunked_gated_delta_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    return kda.load_library()


def header_functions():
    with open(os.path.join(ROOT, "include", "kda.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_\w+)\s*\(", text)))


def test_library_exports_every_header_symbol(lib):
    names = header_functions()
    assert names, "no functions parsed from include/kda.h"
    for n in names:
        assert hasattr(lib, n), f"libkda.so does not export {n}"
    assert set(names) == set(binding.EXPORTS)


def test_status_strings(lib):
    for code in range(8):
        s = kda.status_string(code)
        assert isinstance(s, str) and s
    assert kda.status_string(99) == "unknown status"


def test_chunk_table_matches_flashkda_examples():
    with open(os.path.join(GOLDEN, "flashkda_chunk_table.json")) as f:
        ex = json.load(f)["examples"]
    for e in ex:
        tb, tt, total = kda.chunk_table(e["cu_seqlens"], e["chunk"])
        assert tb == e["tile_base"] and tt == e["t_tiles"]
        assert total == sum(e["t_tiles"])
        if "chunk_lengths" in e:
            L = e["cu_seqlens"][1] - e["cu_seqlens"][0]
            lens = [min(e["chunk"], L - t * e["chunk"]) for t in range(tt[0])]
            assert lens == e["chunk_lengths"]


def test_chunk_table_edge_cases():
    assert kda.chunk_table([0]) == ([], [], 0)
    assert kda.chunk_table([0, 0, 64, 65, 65]) == ([0, 0, 1, 2], [0, 1, 1, 0], 2)
    with pytest.raises(ValueError):
        kda.chunk_table([0, 5, 3])


def test_workspace_size_headline():
    d = kda.make_dims(4, 8192, 32, 128, 128)
    n = kda.workspace_size(d)
    th = 4 * 8192 * 32
    # qg, kg, w, u (4 x 256 B) + Aqk (128 B) + gd (8 B per token-head at 64-token chunks)
    assert 1160 * th <= n <= 1160 * th + (1 << 20)
    L = kda.workspace_layout(d)
    assert L.max_chunks == 4 * 128 and L.chunk == 64 and L.total == n
    offs = [L.status, L.seq_info, L.chunk_info, L.gd, L.qg, L.kg, L.w, L.u, L.aqk, L.total]
    assert offs == sorted(offs)
    for o in (L.gd, L.qg, L.kg, L.w, L.u, L.aqk):
        assert o % 1024 == 0


def test_workspace_size_varlen_bound():
    # sum_s ceil(L_s/64) <= floor((T + 63 N) / 64)
    d = kda.make_dims(1, 1000, 2, 64, 64, num_seqs=7)
    L = kda.workspace_layout(d)
    assert L.max_chunks == (1000 + 63 * 7) // 64
    assert kda.workspace_size(kda.make_dims(1, 10, 2, 96, 64)) == 0  # unsupported K


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on these paths


def call_fwd(lib, dims, q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, cu=None, o=FAKE, ht=None,
             ws=FAKE, ws_bytes=None):
    if ws_bytes is None:
        ws_bytes = 1 << 40
    P = ctypes.c_void_p
    return lib.kda_fwd(P(q), P(k), P(v), P(g), P(beta), 0.1, P(h0), P(cu), P(o), P(ht),
                       ctypes.byref(dims) if dims is not None else None, P(ws), ws_bytes, None)


def test_validation_errors_before_any_launch(lib):
    d = kda.make_dims(1, 128, 2, 128, 128)
    assert call_fwd(lib, None) == 1                                     # NULL dims
    assert call_fwd(lib, kda.make_dims(1, 128, 2, 96, 128)) == 2        # K unsupported
    assert call_fwd(lib, kda.make_dims(1, 128, 2, 128, 192)) == 2       # V unsupported
    assert call_fwd(lib, kda.make_dims(1, -1, 2, 128, 128)) == 1        # negative T
    assert call_fwd(lib, kda.make_dims(1, 128, 0, 128, 128)) == 1       # no heads
    assert call_fwd(lib, d, ws=0) == 4                                  # no workspace
    assert call_fwd(lib, d, ws=FAKE + 64) == 4                          # misaligned workspace
    assert call_fwd(lib, d, ws_bytes=1024) == 4                         # too small
    assert call_fwd(lib, d, q=FAKE + 8) == 3                            # misaligned q
    assert call_fwd(lib, d, g=FAKE + 4) == 3                            # misaligned g
    assert call_fwd(lib, d, k=0) == 1                                   # NULL k
    assert call_fwd(lib, d, cu=FAKE) == 1                               # cu_seqlens without num_seqs
    dv = kda.make_dims(2, 128, 2, 128, 128, num_seqs=3)
    assert call_fwd(lib, dv, cu=FAKE) == 1                              # packed batch needs B == 1
    dv = kda.make_dims(1, 128, 2, 128, 128, num_seqs=3)
    assert call_fwd(lib, dv, cu=None) == 1                              # num_seqs without cu_seqlens
    P = ctypes.c_void_p
    assert lib.kda_selftest_wait_timeout(None, 1000, None) == 1           # no status word
    assert lib.kda_selftest_wait_timeout(P(FAKE + 2), 1000, None) == 1    # misaligned
    assert lib.kda_selftest_wait_timeout(P(FAKE), 0, None) == 1           # no limit
    assert lib.kda_selftest_wait_timeout(P(FAKE), 10**10, None) == 1      # above the kernels' limit


def call_bwd(lib, dims, do=FAKE, dv_in=FAKE, dht=None, dhck=None, dv2=FAKE, dh0=None, ws=FAKE,
             ws_bytes=1 << 40):
    P = ctypes.c_void_p
    return lib.kda_bwd_dh(0.1, P(do), P(dv_in), P(dht), P(dhck), P(dv2), P(dh0),
                          ctypes.byref(dims) if dims is not None else None, P(ws), ws_bytes, None)


def test_bwd_validation_errors_before_any_launch(lib):
    d = kda.make_dims(1, 128, 2, 128, 128)
    assert call_bwd(lib, None) == 1                                     # NULL dims
    assert call_bwd(lib, kda.make_dims(1, 128, 2, 96, 128)) == 2        # K unsupported
    assert call_bwd(lib, d, ws=0) == 4                                  # no workspace
    assert call_bwd(lib, d, ws_bytes=1024) == 4                         # too small
    assert call_bwd(lib, d, do=0) == 1                                  # NULL do
    assert call_bwd(lib, d, dv_in=0) == 1                               # NULL dv_in
    assert call_bwd(lib, d, dv2=0) == 1                                 # NULL dv2
    assert call_bwd(lib, d, do=FAKE + 2) == 3                           # misaligned do
    assert call_bwd(lib, d, dht=FAKE + 4) == 3                          # misaligned dht
    assert call_bwd(lib, d, dh0=FAKE + 8) == 3                          # misaligned dh0


def test_fwd_ex_option_validation(lib):
    P = ctypes.c_void_p
    d = kda.make_dims(1, 128, 4, 128, 128)

    def call(**kw):
        o = kda.FwdOpts(**kw)
        return lib.kda_fwd_ex(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0.1, None, None, P(FAKE), None,
                              ctypes.byref(d), ctypes.byref(o), P(FAKE), 1 << 40, None)

    assert call(io_dtype=2) == 1          # unknown io dtype
    assert call(state_dtype=5) == 1       # unknown state dtype
    assert call(beta_logits=2) == 1       # flag must be 0 / 1
    assert call(qk_heads=3) == 1          # 4 value heads are not a multiple of 3
    assert call(qk_heads=8) == 1          # more q/k heads than value heads
    assert call(qk_heads=-1) == 1
    assert lib.kda_fwd_scan_ex(0.1, None, P(FAKE), None, ctypes.byref(d), ctypes.byref(kda.FwdOpts(io_dtype=7)),
                               P(FAKE), 1 << 40, None) == 1


def test_segmented_scan_plan():
    """The scan is cut into segments only when few (sequence, head, 64-column)
    units would leave most SMs idle over long sequences and the plan's cost
    model expects a gain; the plan depends on the dims alone."""
    lay = kda.workspace_layout(kda.make_dims(4, 8192, 32, 128, 128))     # headline: 256 units
    assert lay.seg_count == 1 and lay.pq == lay.hin == lay.total
    lay = kda.workspace_layout(kda.make_dims(1, 65536, 32, 128, 128))    # long: one wave already
    assert lay.seg_count == 1
    lay = kda.workspace_layout(kda.make_dims(1, 1000, 2, 128, 128))      # too short to cut
    assert lay.seg_count == 1
    cases = [kda.make_dims(1, 65536, 32, 64, 64),                        # long at K = V = 64: 32 units
             kda.make_dims(1, 4096, 16, 128, 128),                       # mid
             kda.make_dims(2, 6405, 1, 64, 64),
             kda.make_dims(1, 10049, 2, 128, 128, num_seqs=5)]           # varlen bound
    for d in cases:
        lay = kda.workspace_layout(d)
        n = d.num_seqs if d.num_seqs > 0 else d.B
        S = lay.seg_count
        assert S >= 2 and lay.seg_len >= 16
        chunks = (d.T + 63) // 64  # every segment holds at least one chunk, together all of them
        assert (S - 1) * lay.seg_len < chunks <= S * lay.seg_len
        assert lay.hin - lay.pq == S * n * d.H * d.K * (d.K + d.V) * 4
        assert lay.total - lay.hin == S * n * d.H * d.K * d.V * 4


def test_staged_forward_plan():
    """One sequence whose scan would leave more than half of the SMs idle, and
    that the segmented plan leaves whole, is run in chunk ranges of at least
    64 chunks (at most 8 ranges); the state passes through the hin region."""
    lay = kda.workspace_layout(kda.make_dims(1, 65536, 32, 128, 128))    # long: 64 scan CTAs
    assert (lay.stage_count, lay.stage_len) == (8, 128)
    assert lay.seg_count == 1 and lay.total - lay.hin == 8 * 32 * 128 * 128 * 4
    lay = kda.workspace_layout(kda.make_dims(1, 12293, 32, 128, 128))    # 193 chunks
    assert (lay.stage_count, lay.stage_len) == (3, 65)
    lay = kda.workspace_layout(kda.make_dims(1, 9000, 32, 128, 128, num_seqs=1))  # one packed sequence
    assert (lay.stage_count, lay.stage_len) == (2, 71)
    for d in [kda.make_dims(4, 8192, 32, 128, 128),           # headline: four sequences
              kda.make_dims(1, 9000, 32, 128, 128, num_seqs=2),
              kda.make_dims(1, 8192, 80, 128, 128),            # 160 scan CTAs: no idle SMs
              kda.make_dims(1, 8000, 32, 128, 128),            # 125 chunks: under two ranges
              kda.make_dims(1, 65536, 32, 64, 64),             # segmented instead
              kda.make_dims(1, 4096, 16, 128, 128)]:           # segmented instead
        lay = kda.workspace_layout(d)
        assert lay.stage_count == 1
    for d in [kda.make_dims(1, 65536, 32, 128, 128), kda.make_dims(1, 8269, 32, 128, 128),
              kda.make_dims(1, 8192, 64, 64, 64)]:
        lay = kda.workspace_layout(d)
        chunks = (d.T + 63) // 64  # every range holds at least one chunk, together all of them
        assert lay.stage_len >= 64 and (lay.stage_count - 1) * lay.stage_len < chunks <= lay.stage_count * lay.stage_len
        assert kda.workspace_size(d) == lay.total


def test_staged_and_host_slice_paths_validate_before_any_launch(lib):
    """The staged forward and the time-slice host pipeline check every argument
    of both stages before anything is enqueued: on this machine (no GPU) any
    launch would fail with KDA_ERR_CUDA, so argument errors must come first."""
    d = kda.make_dims(1, 65536, 32, 128, 128)                           # staged (8 chunk ranges)
    assert kda.workspace_layout(d).stage_count == 8
    assert call_fwd(lib, d, q=FAKE + 8) == 3                            # misaligned q
    assert call_fwd(lib, d, o=0) == 1                                   # no o (a scan-stage argument)
    assert call_fwd(lib, d, o=FAKE + 4) == 3                            # misaligned o
    assert call_fwd(lib, d, ws_bytes=kda.workspace_size(d) - 1) == 4    # one byte short (hin included)
    P = ctypes.c_void_p
    h = kda.make_dims(4, 8192, 32, 128, 128)                            # host pipeline over time slices
    need = kda.host_arena_size(h)
    host = ctypes.create_string_buffer(64)
    args = [P(ctypes.addressof(host))] * 5
    assert lib.kda_fwd_host(*args, ctypes.c_float(0.1), None, None, P(ctypes.addressof(host)), None,
                            ctypes.byref(h), P(FAKE), ctypes.c_size_t(need - 1), None) == 4
    assert lib.kda_fwd_host(*args, ctypes.c_float(0.1), None, None, None, None,
                            ctypes.byref(h), P(FAKE), ctypes.c_size_t(need), None) == 1  # no o


def test_workspace_regions_hold_what_the_kernels_write():
    """For a seeded spread of shapes (fixed length and packed, K and V of 64 and
    128, short to long, few to many heads), the workspace regions are aligned,
    in order, disjoint, and each is at least as large as what the kernels
    index in it: the chunk table, gd, qg, kg, w, u, Aqk per (chunk, head)
    tile, the segment maps [P | Q], and the entry states of the segments or
    the chunk ranges of the staged forward."""
    import random
    rng = random.Random(20261202)
    cases = [(4, 8192, 32, 128, 128, 0), (1, 65536, 32, 128, 128, 0), (1, 65536, 32, 64, 64, 0),
             (1, 4096, 16, 128, 128, 0), (1, 9000, 32, 128, 128, 1), (1, 10049, 2, 128, 128, 5)]
    for _ in range(200):
        K, V = rng.choice((64, 128)), rng.choice((64, 128))
        if rng.random() < 0.5:
            cases.append((rng.randint(1, 8), rng.randint(0, 40000), rng.randint(1, 96), K, V, 0))
        else:
            n = rng.randint(1, 40)
            cases.append((1, rng.randint(0, 60000), rng.randint(1, 96), K, V, n))
    for B, T, H, K, V, ns in cases:
        d = kda.make_dims(B, T, H, K, V, ns)
        L = kda.workspace_layout(d)
        names = ["status", "seq_info", "chunk_info", "gd", "qg", "kg", "w", "u", "aqk", "pq", "hin", "total"]
        offs = [getattr(L, n) for n in names]
        assert offs == sorted(offs), (B, T, H, K, V, ns)
        assert all(o % 256 == 0 for o in offs[:3]) and all(o % 1024 == 0 for o in offs[3:-1])
        N = ns if ns > 0 else B
        nc = L.max_chunks
        assert nc == ((T + 63 * N) // 64 if ns > 0 else B * ((T + 63) // 64))
        tiles = nc * H
        need = {"seq_info": 16 * max(N, 1), "chunk_info": 8 * max(nc, 1), "gd": tiles * K * 4,
                "qg": tiles * 64 * K * 2, "kg": tiles * 64 * K * 2, "w": tiles * 64 * K * 2,
                "u": tiles * 64 * V * 2, "aqk": tiles * 64 * 64 * 2}
        for i, n in enumerate(names[1:-3], start=1):
            assert offs[i + 1] - offs[i] >= need[n], (n, B, T, H, K, V, ns)
        seg_units = L.seg_count * N * H if L.seg_count > 1 else 0
        stage_units = L.stage_count * N * H if L.stage_count > 1 else 0
        assert L.hin - L.pq >= seg_units * K * (K + V) * 4
        assert L.total - L.hin >= max(seg_units, stage_units) * K * V * 4
        assert not (L.seg_count > 1 and L.stage_count > 1)
        if L.stage_count > 1:
            assert N == 1 and (L.stage_count - 1) * L.stage_len < (T + 63) // 64 <= L.stage_count * L.stage_len
        assert kda.workspace_size(d) == L.total


def test_noalloc_capacity_and_plan():
    """kda_fwd_noalloc runs the two stages on the caller's stream; kda_fwd would
    run a staged plan (library streams) only for problems whose workspace far
    exceeds the scratch array, so within the scratch capacity both entry
    points take the same plan.  Also pins the capacity the header states."""
    cap = kda.binding.NOALLOC_SCRATCH_BYTES

    def fits(B, T, H, K, V, n=0):
        s = kda.workspace_size(kda.make_dims(B, T, H, K, V, n))
        return 0 < s <= cap

    assert fits(1, 53248, 1, 128, 128) and not fits(1, 53249, 1, 128, 128)
    assert fits(1, 1792, 32, 128, 128) and not fits(1, 1793, 32, 128, 128)
    for H in (1, 2, 3, 8, 16, 24, 32, 48, 64, 128):
        for K, V in ((128, 128), (64, 64), (128, 64), (64, 128)):
            for T in list(range(1, 110000, 1777)) + [53248, 101376]:
                for d in (kda.make_dims(1, T, H, K, V), kda.make_dims(1, T, H, K, V, 1)):
                    s = kda.workspace_size(d)
                    if 0 < s <= cap:
                        assert kda.workspace_layout(d).stage_count == 1, (T, H, K, V)


def test_context_parallel_entries_validate_before_any_launch(lib):
    """kda_fwd_state_map and kda_chain_states reject bad arguments before any
    driver call (on this machine a launch would fail with KDA_ERR_CUDA)."""
    P = ctypes.c_void_p
    d = kda.make_dims(2, 130, 2, 128, 128)

    def smap(dims=d, q=FAKE, pq=FAKE, ws=FAKE, ws_bytes=1 << 40):
        return lib.kda_fwd_state_map(P(q), P(FAKE), P(FAKE), P(FAKE), P(FAKE), None, P(pq),
                                     ctypes.byref(dims) if dims is not None else None, P(ws), ws_bytes, None)

    assert smap(dims=None) == 1                                       # NULL dims
    assert smap(dims=kda.make_dims(2, 130, 2, 96, 128)) == 2          # K unsupported
    assert smap(pq=0) == 1                                            # no output
    assert smap(pq=FAKE + 8) == 3                                     # misaligned output
    assert smap(q=FAKE + 2) == 3                                      # misaligned q
    assert smap(ws_bytes=1024) == 4                                   # workspace too small

    def chain(pq=FAKE, h0=None, h_in=FAKE, R=2, N=2, H=2, K=128, V=128):
        return lib.kda_chain_states(P(pq), P(h0), P(h_in), R, N, H, K, V, None)

    assert chain(R=0) == 1 and chain(N=-1) == 1 and chain(H=0) == 1   # counts
    assert chain(K=96) == 2 and chain(V=32) == 2                      # unsupported dims
    assert chain(pq=0) == 1 and chain(h_in=0) == 1                    # NULL pointers
    assert chain(pq=FAKE + 4) == 3 and chain(h0=FAKE + 4) == 3        # misaligned
    assert chain(N=0) == 0                                            # nothing to do


def test_fused_plan_options_validate_before_any_launch(lib):
    """The plan option: unknown values are rejected, the single-pass kernel with
    an interface variant is unsupported, both before any driver call; the
    automatic plan takes the two stages (on this machine it then fails at its
    first driver call, KDA_ERR_CUDA)."""
    P = ctypes.c_void_p
    d = kda.make_dims(1, 128, 2, 128, 128)

    def fwd_ex(**kw):
        o = kda.FwdOpts(**kw)
        return lib.kda_fwd_ex(P(FAKE), P(FAKE), P(FAKE), P(FAKE), P(FAKE), 0.1, None, None, P(FAKE), None,
                              ctypes.byref(d), ctypes.byref(o), P(FAKE), 1 << 40, None)

    assert fwd_ex(plan=3) == 1 and fwd_ex(plan=-1) == 1
    assert fwd_ex(plan=2, io_dtype=1) == 2 and fwd_ex(plan=2, beta_logits=1) == 2
    assert fwd_ex(plan=2, state_dtype=1) == 2 and fwd_ex(plan=2, qk_heads=1) == 2
    assert fwd_ex(plan=0, io_dtype=1) == 5 and fwd_ex(plan=1) == 5
