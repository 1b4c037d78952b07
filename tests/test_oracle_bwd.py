"""Pins of the fp64 reverse state scan (oracle/chunked.chunk_bwd_dh) against
computations that do not share its formula: the token-level adjoint of the
recurrence (for the state gradients) and finite differences of the chunked
forward (for dv2, the gradient with respect to a chunk's v')."""
import numpy as np
import pytest

from oracle import chunked


def rand(rng, L, K, V, mu=1.0):
    q = rng.standard_normal((L, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((L, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((L, V))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    g = -np.log1p(np.exp(-(rng.standard_normal((L, K)) + mu)))
    return q, k, v, g, beta


def token_adjoint(q, k, g, beta, scale, do, dht, boundaries):
    """Reverse-mode through S_t = (I - b k k^T) D_t S_{t-1} + b k v^T, o_t = scale S_t^T q_t,
    for the loss sum(do * o) + sum(dht * S_T): returns dS at the requested token
    boundaries (dS_t = gradient w.r.t. the state after token t)."""
    L, K = q.shape
    dS = np.array(dht, dtype=np.float64, copy=True)
    out = {}
    for t in range(L, 0, -1):
        if t in boundaries:
            out[t] = dS.copy()
        i = t - 1
        dS = dS + scale * np.outer(q[i], do[i])
        # adjoint of X -> (I - b k k^T) D X  is  Y -> D (I - b k k^T) Y
        P = np.eye(K) - beta[i] * np.outer(k[i], k[i])
        dS = np.exp(g[i])[:, None] * (P @ dS)
    out[0] = dS
    return out


@pytest.mark.parametrize("L", [1, 64, 65, 150])
def test_state_gradients_match_token_adjoint(L):
    rng = np.random.default_rng(L)
    K, V, C, scale = 8, 5, 16, 0.4
    q, k, v, g, beta = rand(rng, L, K, V)
    do = rng.standard_normal((L, V))
    dht = rng.standard_normal((K, V))
    chunks = chunked.chunk_intra(q, k, v, g, beta, scale, C)
    # the full v' gradient includes the chunk-local Aqk^T do term: pass it as dv_in
    dv_in = np.zeros((L, V))
    for c, ch in enumerate(chunks):
        a = c * C
        n = ch["valid"]
        dv_in[a:a + n] = (ch["Aqk"].T @ np.vstack([do[a:a + n], np.zeros((C - n, V))]))[:n]
    dhck, dv2, dh0 = chunked.chunk_bwd_dh(chunks, do, dv_in, dht, scale)
    bounds = {min((c + 1) * C, L) for c in range(len(chunks))}
    ref = token_adjoint(q, k, g, beta, scale, do, dht, bounds)
    for c in range(len(chunks)):
        np.testing.assert_allclose(dhck[c], ref[min((c + 1) * C, L)], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dh0, ref[0], rtol=1e-10, atol=1e-12)


def test_dv2_is_the_vprime_gradient_by_finite_differences():
    """L = sum(do*o) + sum(dht*ht) is linear in one chunk's v' (h0 and the
    other inputs fixed), so a finite difference is exact up to rounding."""
    rng = np.random.default_rng(7)
    L, K, V, C, scale = 100, 8, 4, 32, 0.6
    q, k, v, g, beta = rand(rng, L, K, V)
    h0 = rng.standard_normal((K, V))
    do = rng.standard_normal((L, V))
    dht = rng.standard_normal((K, V))
    chunks = chunked.chunk_intra(q, k, v, g, beta, scale, C)
    dv_in = np.zeros((L, V))
    for c, ch in enumerate(chunks):
        a, n = c * C, ch["valid"]
        dv_in[a:a + n] = (ch["Aqk"].T @ np.vstack([do[a:a + n], np.zeros((C - n, V))]))[:n]
    _, dv2, _ = chunked.chunk_bwd_dh(chunks, do, dv_in, dht, scale)

    def loss(override):
        o, ht = chunked.scan_with_vprime(chunks, h0, scale, override)
        return float(np.sum(do * o) + np.sum(dht * ht))

    base = loss(None)
    for c in range(len(chunks)):
        n = chunks[c]["valid"]
        E = np.zeros((C, V))
        E[:n] = rng.standard_normal((n, V))
        fd = loss((c, E)) - base
        np.testing.assert_allclose(fd, np.sum(dv2[c * C:c * C + n] * E[:n]), rtol=1e-9, atol=1e-9)


def test_dh0_is_the_h0_gradient_by_finite_differences():
    rng = np.random.default_rng(8)
    L, K, V, C, scale = 70, 6, 3, 16, 0.3
    q, k, v, g, beta = rand(rng, L, K, V)
    h0 = rng.standard_normal((K, V))
    do = rng.standard_normal((L, V))
    dht = rng.standard_normal((K, V))
    chunks = chunked.chunk_intra(q, k, v, g, beta, scale, C)
    dv_in = np.zeros((L, V))
    for c, ch in enumerate(chunks):
        a, n = c * C, ch["valid"]
        dv_in[a:a + n] = (ch["Aqk"].T @ np.vstack([do[a:a + n], np.zeros((C - n, V))]))[:n]
    _, _, dh0 = chunked.chunk_bwd_dh(chunks, do, dv_in, dht, scale)

    def loss(h):
        o, ht = chunked.scan_with_vprime(chunks, h, scale)
        return float(np.sum(do * o) + np.sum(dht * ht))

    E = rng.standard_normal((K, V))
    np.testing.assert_allclose(loss(h0 + E) - loss(h0), np.sum(dh0 * E), rtol=1e-9, atol=1e-9)


def test_varlen_bwd_equals_separate_sequences():
    rng = np.random.default_rng(9)
    lengths = [30, 0, 70]
    T, H, K, V = sum(lengths), 2, 8, 4
    q = rng.standard_normal((1, T, H, K)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((1, T, H, K)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, H, V))
    g = -np.log1p(np.exp(-(rng.standard_normal((1, T, H, K)) + 1)))
    beta = 1 / (1 + np.exp(-rng.standard_normal((1, T, H))))
    do = rng.standard_normal((1, T, H, V))
    dvi = rng.standard_normal((1, T, H, V))
    dht = rng.standard_normal((3, H, K, V))
    cu = np.concatenate([[0], np.cumsum(lengths)])
    dhck, dv2, dh0 = chunked.chunked_bwd_dh(q, k, v, g, beta, 0.5, do, dvi, dht=dht, cu_seqlens=cu, C=64)
    np.testing.assert_array_equal(dh0[1], dht[1])  # empty sequence
    off = 0
    for s, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if b == a:
            continue
        ck, d2, d0 = chunked.chunked_bwd_dh(q[:, a:b], k[:, a:b], v[:, a:b], g[:, a:b], beta[:, a:b], 0.5,
                                            do[:, a:b], dvi[:, a:b], dht=dht[s:s + 1], C=64)
        n = ck.shape[0]
        np.testing.assert_allclose(dhck[off:off + n], ck, rtol=1e-12)
        np.testing.assert_allclose(dv2[:, a:b], d2, rtol=1e-12)
        np.testing.assert_allclose(dh0[s], d0[0], rtol=1e-12)
        off += n
