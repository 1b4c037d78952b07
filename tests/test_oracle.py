"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test fixes the oracle to a closed form, an invariant, a hand-worked
example, or the independently written chunked form, so that a dropped term,
a wrong sign or index, the wrong decay/delta order, or beta on the wrong side
fails at least one of them.  CPU only.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def rand_inputs(rng, B, T, H, K, V, mu=2.0, h0=True):
    q = rng.standard_normal((B, T, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H))))
    x = rng.standard_normal((B, T, H, K)) + mu
    g = -np.log1p(np.exp(-x))  # logsigmoid
    hh = 0.1 * rng.standard_normal((B, H, K, V)) if h0 else None
    return q, k, v, g, beta, hh


def rec(q, k, v, g, beta, scale, h0=None, cu=None, **kw):
    return oracle.recurrent_fwd(q, k, v, g, beta, scale, h0=h0, cu_seqlens=cu,
                                fp64_inputs=True, **kw)


# ---------------------------------------------------------------- closed forms

def test_beta0_g0_state_is_h0():
    """beta = 0 and g = 0: nothing is written or decayed, S_t = h0, o = scale h0^T q."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 2, 9, 3, 8, 5)
    g[:] = 0.0
    beta[:] = 0.0
    o, ht = rec(q, k, v, g, beta, 0.7, h0)
    np.testing.assert_array_equal(ht, h0)
    want = 0.7 * np.einsum("bthd,bhdv->bthv", q, h0)
    np.testing.assert_allclose(o, want, rtol=1e-13, atol=1e-15)


def test_beta0_decay_only_closed_form():
    """beta = 0: S_t = Diag(exp(sum_{s<=t} g_s)) h0 (decay is per key row, inclusive)."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 1, 11, 2, 6, 4, mu=0.5)
    beta[:] = 0.0
    o, ht = rec(q, k, v, g, beta, 1.3, h0)
    cum = np.cumsum(g, axis=1)  # [B,T,H,K]
    St = np.exp(cum)[..., None] * h0[:, None]  # [B,T,H,K,V]
    want_o = 1.3 * np.einsum("bthd,bthdv->bthv", q, St)
    np.testing.assert_allclose(o, want_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(ht, St[:, -1], rtol=1e-12, atol=1e-14)


def test_full_forget_stores_last_pair():
    """g = -inf, beta = 1: the state forgets everything, S_t = k_t v_t^T and o_t = scale (q_t.k_t) v_t."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 1, 7, 2, 8, 5)
    g[:] = -np.inf
    beta[:] = 1.0
    o, ht = rec(q, k, v, g, beta, 0.5, h0)
    want_o = 0.5 * np.einsum("bthd,bthd->bth", q, k)[..., None] * v
    np.testing.assert_allclose(o, want_o, rtol=1e-12, atol=1e-14)
    want_ht = np.einsum("bhd,bhv->bhdv", k[:, -1], v[:, -1])
    np.testing.assert_allclose(ht, want_ht, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("T", [5, 8])
def test_orthonormal_keys_recall(T):
    """beta = 1, g = 0, orthonormal keys: ht = (I - sum k k^T) h0 + sum k v^T, and ht^T k_j = v_j."""
    K, V = 8, 6
    Qm, _ = np.linalg.qr(RNG.standard_normal((K, K)))
    k = Qm[:, :T].T.reshape(1, T, 1, K).copy()  # rows are orthonormal keys
    q = RNG.standard_normal((1, T, 1, K))
    v = RNG.standard_normal((1, T, 1, V))
    g = np.zeros((1, T, 1, K))
    beta = np.ones((1, T, 1))
    h0 = RNG.standard_normal((1, 1, K, V))
    _, ht = rec(q, k, v, g, beta, 1.0, h0)
    kk = k[0, :, 0]  # [T, K]
    P = np.eye(K) - kk.T @ kk
    want = P @ h0[0, 0] + kk.T @ v[0, :, 0]
    np.testing.assert_allclose(ht[0, 0], want, rtol=1e-12, atol=1e-12)
    recall = ht[0, 0].T @ kk.T  # [V, T]
    np.testing.assert_allclose(recall.T, v[0, :, 0], rtol=1e-12, atol=1e-12)


def test_overwrite_same_key():
    """Writing (k, v1) then (k, v2) with beta = 1, g = 0 and |k| = 1 leaves S^T k = v2."""
    K, V = 5, 3
    kv = RNG.standard_normal(K)
    kv /= np.linalg.norm(kv)
    k = np.stack([kv, kv]).reshape(1, 2, 1, K)
    v = RNG.standard_normal((1, 2, 1, V))
    q = np.stack([kv, kv]).reshape(1, 2, 1, K)
    g = np.zeros((1, 2, 1, K))
    beta = np.ones((1, 2, 1))
    h0 = RNG.standard_normal((1, 1, K, V))
    o, ht = rec(q, k, v, g, beta, 1.0, h0)
    np.testing.assert_allclose(ht[0, 0].T @ kv, v[0, 1, 0], rtol=1e-12, atol=1e-12)
    # reading with q = k right after each write returns the value just written
    np.testing.assert_allclose(o[0, :, 0], v[0, :, 0], rtol=1e-12, atol=1e-12)


def test_scalar_constant_coefficients_closed_form():
    """K = V = 1 with constant inputs: s_t = a s_{t-1} + b, a = (1 - beta k^2) e^g, b = beta k v,
    so s_t = a^t s_0 + b (1 - a^t) / (1 - a)."""
    T = 37
    kk, vv, bb, gg, qq, s0, sc = 0.8, -1.7, 0.6, -0.05, 1.4, 0.9, 0.3
    q = np.full((1, T, 1, 1), qq)
    k = np.full((1, T, 1, 1), kk)
    v = np.full((1, T, 1, 1), vv)
    g = np.full((1, T, 1, 1), gg)
    beta = np.full((1, T, 1), bb)
    h0 = np.full((1, 1, 1, 1), s0)
    o, ht = rec(q, k, v, g, beta, sc, h0)
    a = (1 - bb * kk * kk) * np.exp(gg)
    b = bb * kk * vv
    t = np.arange(1, T + 1)
    s = a ** t * s0 + b * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(o[0, :, 0, 0], sc * qq * s, rtol=1e-12)
    np.testing.assert_allclose(ht[0, 0, 0, 0], s[-1], rtol=1e-12)


def test_hand_worked_2x2():
    """A two-token K = V = 2 example worked by hand (tests/golden/hand_2x2.json)."""
    with open(os.path.join(GOLDEN, "hand_2x2.json")) as f:
        ex = json.load(f)
    q = np.array(ex["q"]).reshape(1, 2, 1, 2)
    k = np.array(ex["k"]).reshape(1, 2, 1, 2)
    v = np.array(ex["v"]).reshape(1, 2, 1, 2)
    g = np.log(np.array(ex["g_exp"])).reshape(1, 2, 1, 2)
    beta = np.array(ex["beta"]).reshape(1, 2, 1)
    h0 = np.array(ex["h0"]).reshape(1, 1, 2, 2)
    o, ht = rec(q, k, v, g, beta, ex["scale"], h0)
    np.testing.assert_allclose(o[0, :, 0], np.array(ex["o"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht[0, 0], np.array(ex["ht"]), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- invariants

def test_linear_in_v_and_h0_exactly():
    """(v, h0) -> (o, S) is linear: doubling both doubles o and ht bit for bit."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 2, 13, 2, 8, 4)
    o1, h1 = rec(q, k, v, g, beta, 0.35, h0)
    o2, h2 = rec(q, k, 2 * v, g, beta, 0.35, 2 * h0)
    np.testing.assert_array_equal(o2, 2 * o1)
    np.testing.assert_array_equal(h2, 2 * h1)


def test_causal():
    """Changing tokens after t leaves o[:t+1] unchanged."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 1, 20, 2, 6, 5)
    o1, _ = rec(q, k, v, g, beta, 0.4, h0)
    k2, v2 = k.copy(), v.copy()
    k2[:, 12:] = RNG.standard_normal(k2[:, 12:].shape)
    v2[:, 12:] += 3.0
    o2, _ = rec(q, k2, v2, g, beta, 0.4, h0)
    np.testing.assert_array_equal(o1[:, :12], o2[:, :12])
    assert not np.allclose(o1[:, 12:], o2[:, 12:])


def test_varlen_equals_separate_runs_and_empty_sequence():
    lengths = [5, 0, 17, 64, 1]
    T = sum(lengths)
    H, K, V = 2, 8, 4
    q, k, v, g, beta, _ = rand_inputs(RNG, 1, T, H, K, V)
    h0 = RNG.standard_normal((len(lengths), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, ht = rec(q, k, v, g, beta, 0.6, h0, cu)
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        sl = slice(a, b)
        os_, hs = rec(q[:, sl], k[:, sl], v[:, sl], g[:, sl], beta[:, sl], 0.6, h0[s:s + 1])
        np.testing.assert_array_equal(o[:, sl], os_)
        np.testing.assert_array_equal(ht[s], hs[0])
    np.testing.assert_array_equal(ht[1], h0[1])  # empty sequence: ht = h0


def test_state_continuation():
    """run(T1 + T2) equals run(T2) started from run(T1)'s final state."""
    q, k, v, g, beta, h0 = rand_inputs(RNG, 1, 30, 2, 6, 3)
    o, ht = rec(q, k, v, g, beta, 0.9, h0)
    oa, ha = rec(q[:, :11], k[:, :11], v[:, :11], g[:, :11], beta[:, :11], 0.9, h0)
    ob, hb = rec(q[:, 11:], k[:, 11:], v[:, 11:], g[:, 11:], beta[:, 11:], 0.9, ha)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(hb, ht, rtol=1e-13, atol=1e-15)


def test_units_subset_and_threads_do_not_change_results():
    q, k, v, g, beta, h0 = rand_inputs(RNG, 2, 19, 3, 8, 4)
    o, ht = rec(q, k, v, g, beta, 0.5, h0, nthreads=1)
    o4, ht4 = rec(q, k, v, g, beta, 0.5, h0, nthreads=4)
    np.testing.assert_array_equal(o, o4)
    np.testing.assert_array_equal(ht, ht4)
    os_, hs = rec(q, k, v, g, beta, 0.5, h0, units=[(1, 2), (0, 0)])
    np.testing.assert_array_equal(os_[1, :, 2], o[1, :, 2])
    np.testing.assert_array_equal(os_[0, :, 0], o[0, :, 0])
    assert np.isnan(os_[0, :, 1]).all()
    np.testing.assert_array_equal(hs[1, 2], ht[1, 2])


def test_bf16_entry_widens_exactly():
    """The bf16/fp32 entry point equals the fp64 entry point on the widened values."""
    torch = pytest.importorskip("torch")
    from chunked_gated_delta_gb300 import synth
    w = synth.Workload("t", B=1, T=70, H=2, K=16, V=8, seed=5)
    x = synth.make_inputs(w)
    o1, h1 = oracle.recurrent_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["scale"],
                                  h0=x["h0"])
    f = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    o2, h2 = rec(f(x["q"]), f(x["k"]), f(x["v"]), f(x["g"]), f(x["beta"]), x["scale"],
                 f(x["h0"]))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(h1, h2)


# ---------------------------------------------------------------- chunked == recurrent

@pytest.mark.parametrize("C", [1, 16, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200])
def test_chunked_equals_recurrent(C, T):
    """The chunked form (independently written, numpy) agrees with the C recurrence to 1e-10."""
    rng = np.random.default_rng(1000 * C + T)
    q, k, v, g, beta, h0 = rand_inputs(rng, 1, T, 2, 16, 8, mu=1.0)
    o_r, h_r = rec(q, k, v, g, beta, 0.25, h0)
    o_c, h_c = chunked.chunked_fwd(q, k, v, g, beta, 0.25, h0, C=C)
    err_o = np.linalg.norm(o_c - o_r) / np.linalg.norm(o_r)
    err_h = np.linalg.norm(h_c - h_r) / np.linalg.norm(h_r)
    assert err_o < 1e-10 and err_h < 1e-10, (err_o, err_h)


def test_chunked_equals_recurrent_varlen_strong_decay():
    """Varlen packing plus decays strong enough that a single in-chunk reference would overflow."""
    rng = np.random.default_rng(77)
    lengths = [70, 3, 0, 129]
    T = sum(lengths)
    q, k, v, g, beta, _ = rand_inputs(rng, 1, T, 2, 8, 4, mu=-6.0)  # g ~ -6 per token
    h0 = rng.standard_normal((len(lengths), 2, 8, 4))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    o_r, h_r = rec(q, k, v, g, beta, 0.5, h0, cu.astype(np.int32))
    o_c, h_c = chunked.chunked_fwd(q, k, v, g, beta, 0.5, h0, cu_seqlens=cu, C=64)
    assert np.all(np.isfinite(o_c))
    np.testing.assert_allclose(o_c, o_r, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(h_c, h_r, rtol=1e-10, atol=1e-12)


def test_chunk_intra_structure():
    """Structural facts of the intra stage: Aqk is zero above the diagonal, A strictly lower,
    T unit lower triangular with (I + A) T = I, and a tail chunk's padded rows are inert."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, _ = rand_inputs(rng, 1, 50, 1, 8, 4)
    ch = chunked.chunk_intra(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0],
                             0.5, C=64)
    assert len(ch) == 1 and ch[0]["valid"] == 50
    c = ch[0]
    assert np.all(np.triu(c["Aqk"], 1) == 0)
    assert np.all(np.triu(c["A"]) == 0)
    np.testing.assert_allclose((np.eye(64) + c["A"]) @ c["T"], np.eye(64), atol=1e-12)
    assert np.all(np.diag(c["T"]) == 1) and np.all(np.triu(c["T"], 1) == 0)
    np.testing.assert_allclose(c["G"], c["g2"][49], rtol=0, atol=0)
    assert np.all(c["w"][50:] == 0) and np.all(c["u"][50:] == 0)
    # log2-space cumsum: exp2(G) equals the product of exp(g) over the chunk
    np.testing.assert_allclose(np.exp2(c["G"]), np.exp(np.sum(g[0, :, 0], axis=0)), rtol=1e-12)
