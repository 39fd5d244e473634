"""The recurrence properties the oracle must satisfy, exactly in fp64 (to
<= 1e-12 where rounding order differs):

(a) unit-norm k, beta=1, g=0  =>  S' k = v
(b) beta=0, g=0               =>  S' = S bitwise
(c) whole segment == the same segment split at any token (state and outputs)
(d) chunk-wise summation (any chunk length) == token-by-token recurrence
(e) brute-force matrix expansion == the recurrence on small D
plus index-orientation and closed-form checks of the recurrence itself.
"""

import numpy as np
import pytest

import oracle


def _rand_case(seed, T, Hk, Hv, D, g_scale=0.3, s_scale=0.2):
    rng = np.random.default_rng(seed)
    q = oracle.l2norm(rng.normal(size=(T, Hk, D)))
    k = oracle.l2norm(rng.normal(size=(T, Hk, D)))
    v = rng.normal(size=(T, Hv, D))
    g = -np.abs(rng.normal(size=(T, Hv))) * g_scale
    beta = rng.uniform(0.05, 0.95, size=(T, Hv))
    S = rng.normal(size=(Hv, D, D)) * s_scale
    return q, k, v, g, beta, S


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


@pytest.mark.parametrize("mp", [oracle.GROUPED, oracle.TILED])
def test_a_unit_key_full_write(mp):
    rng = np.random.default_rng(1)
    Hk, Hv, D = 2, 4, 16
    q, k, v, _, _, S = _rand_case(2, 1, Hk, Hv, D)
    k = rng.normal(size=(1, Hk, D))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)  # unit norm to fp64 rounding
    g = np.zeros((1, Hv))
    beta = np.ones((1, Hv))
    _, S1 = oracle.delta(q, k, v, g, beta, S, mp)
    for h in range(Hv):
        kh = oracle.k_head(mp, h, Hk, Hv)
        Sk = S1[h] @ k[0, kh]
        assert np.max(np.abs(Sk - v[0, h])) < 1e-12
    del rng


def test_b_no_write_no_decay_is_identity():
    q, k, v, _, _, S = _rand_case(3, 6, 2, 6, 8)
    g = np.zeros((6, 6))
    beta = np.zeros((6, 6))
    o, S1 = oracle.delta(q, k, v, g, beta, S, oracle.GROUPED)
    assert np.array_equal(S1, S)
    # the output then is just the scaled read-out of the untouched state
    for t in range(6):
        for h in range(6):
            kh = oracle.k_head(oracle.GROUPED, h, 2, 6)
            ref = S[h] @ q[t, kh] / np.sqrt(8)
            assert np.max(np.abs(o[t, h] - ref)) < 1e-14


@pytest.mark.parametrize("split", [0, 1, 3, 17, 63, 64, 65, 100])
def test_c_split_anywhere(split):
    T = 101
    q, k, v, g, beta, S = _rand_case(4, T, 2, 4, 16)
    o, S1 = oracle.delta(q, k, v, g, beta, S, oracle.TILED)
    oa, Sa = oracle.delta(q[:split], k[:split], v[:split], g[:split], beta[:split], S, oracle.TILED)
    ob, Sb = oracle.delta(q[split:], k[split:], v[split:], g[split:], beta[split:], Sa,
                          oracle.TILED)
    assert np.array_equal(np.concatenate([oa, ob]), o)
    assert np.array_equal(Sb, S1)


def test_c_split_segment_with_conv_state():
    rng = np.random.default_rng(9)
    Hk, Hv, D, T = 2, 4, 8, 9
    C = 2 * Hk * D + Hv * D
    x = rng.normal(size=(T, C))
    a, b, z = rng.normal(size=(T, Hv)), rng.normal(size=(T, Hv)), rng.normal(size=(T, Hv, D))
    w = rng.normal(size=(C, 4)) * 0.4
    A_log, dt = np.log(rng.uniform(1, 4, Hv)), rng.uniform(-0.5, 0.5, Hv)
    nw = rng.uniform(0.8, 1.2, D)
    cs, S = rng.normal(size=(C, 3)), rng.normal(size=(Hv, D, D)) * 0.1
    args = (Hk, Hv, D, oracle.GROUPED, oracle.LOG_RATE)
    full = oracle.segment(*args, x, a, b, z, w, A_log, dt, nw, cs, S)
    for split in (1, 2, 3, 5, 8):
        p1 = oracle.segment(*args, x[:split], a[:split], b[:split], z[:split], w, A_log, dt, nw,
                            cs, S)
        p2 = oracle.segment(*args, x[split:], a[split:], b[split:], z[split:], w, A_log, dt, nw,
                            p1[2], p1[3])
        assert np.array_equal(np.concatenate([p1[0], p2[0]]), full[0])
        assert np.array_equal(np.concatenate([p1[1], p2[1]]), full[1])
        assert np.array_equal(p2[2], full[2])
        assert np.array_equal(p2[3], full[3])


@pytest.mark.parametrize("chunk", [1, 7, 64, 145])
@pytest.mark.parametrize("g_scale", [0.02, 0.5, 8.0])
def test_d_chunked_equals_recurrence(chunk, g_scale):
    T = 145
    q, k, v, g, beta, S = _rand_case(5, T, 2, 4, 16, g_scale=g_scale)
    for mp in (oracle.GROUPED, oracle.TILED):
        o, S1 = oracle.delta(q, k, v, g, beta, S, mp)
        oc, Sc = oracle.delta_chunked(q, k, v, g, beta, S, mp, chunk)
        assert np.max(np.abs(oc - o)) < 1e-12 * max(1.0, np.max(np.abs(o)))
        assert np.max(np.abs(Sc - S1)) < 1e-12 * max(1.0, np.max(np.abs(S1)))


def test_d_chunked_underflowing_decay():
    """g down to -50 per token: the cumulative decay underflows fp64 inside a
    chunk; the chunked form must still agree (it never divides by e^{c})."""
    T = 70
    q, k, v, g, beta, S = _rand_case(6, T, 1, 2, 8)
    g = -np.random.default_rng(0).uniform(0, 50, size=(T, 2))
    o, S1 = oracle.delta(q, k, v, g, beta, S, oracle.GROUPED)
    oc, Sc = oracle.delta_chunked(q, k, v, g, beta, S, oracle.GROUPED, 64)
    assert np.all(np.isfinite(oc)) and np.all(np.isfinite(Sc))
    assert np.max(np.abs(oc - o)) < 1e-12 and np.max(np.abs(Sc - S1)) < 1e-12


@pytest.mark.parametrize("mp", [oracle.GROUPED, oracle.TILED])
def test_e_bruteforce_d4(mp):
    T = 23
    q, k, v, g, beta, S = _rand_case(7, T, 2, 4, 4, g_scale=0.4, s_scale=0.5)
    o, S1 = oracle.delta(q, k, v, g, beta, S, mp)
    ob, Sb = oracle.delta_bruteforce(q, k, v, g, beta, S, mp)
    assert np.max(np.abs(ob - o)) < 1e-12
    assert np.max(np.abs(Sb - S1)) < 1e-12


def test_e_bruteforce_unnormalised_keys():
    """With keys of norm != 1 the rank-one update no longer projects; the
    expansion S(I - b k k^T) still has to match."""
    rng = np.random.default_rng(8)
    T, Hk, Hv, D = 9, 1, 2, 4
    q, k = rng.normal(size=(T, Hk, D)), rng.normal(size=(T, Hk, D)) * 0.7
    v, S = rng.normal(size=(T, Hv, D)), rng.normal(size=(Hv, D, D))
    g, beta = -rng.uniform(0, 1, (T, Hv)), rng.uniform(0, 1, (T, Hv))
    o, S1 = oracle.delta(q, k, v, g, beta, S, oracle.GROUPED)
    ob, Sb = oracle.delta_bruteforce(q, k, v, g, beta, S, oracle.GROUPED)
    assert _rel(ob, o) < 1e-12 and _rel(Sb, S1) < 1e-12


def test_scalar_closed_form_with_decay():
    """D=1: S' = a S + b (v - a S k) k and o = S' q (scale 1)."""
    rng = np.random.default_rng(10)
    for _ in range(20):
        S0, q, k, v = rng.normal(size=4)
        g, b = -abs(rng.normal()), rng.uniform()
        o, S1 = oracle.delta(np.array([[[q]]]), np.array([[[k]]]), np.array([[[v]]]),
                             np.array([[g]]), np.array([[b]]), np.array([[[S0]]]), 0)
        a = np.exp(g)
        Sr = a * S0 + b * (v - a * S0 * k) * k
        assert abs(S1.ravel()[0] - Sr) < 1e-14 * max(1, abs(Sr))
        assert abs(o.ravel()[0] - Sr * q) < 1e-14 * max(1, abs(Sr * q))


def test_state_orientation_value_row_key_column():
    """S[h][j][i]: j indexes the value (output) row, i the key. A one-hot state
    at (j0, i0) read with q = e_{i0} lights output j0 only."""
    Hk, Hv, D = 1, 1, 8
    j0, i0 = 5, 2
    S = np.zeros((Hv, D, D))
    S[0, j0, i0] = 1.0
    q = np.zeros((1, Hk, D))
    q[0, 0, i0] = 1.0
    k = np.zeros((1, Hk, D))
    k[0, 0, 7] = 1.0
    v = np.zeros((1, Hv, D))
    o, S1 = oracle.delta(q, k, v, np.zeros((1, 1)), np.zeros((1, 1)), S, 0)
    expect = np.zeros(D)
    expect[j0] = 1.0 / np.sqrt(D)
    assert np.array_equal(o[0, 0], expect)
    # one write with beta=1, g=0 from zero state: S = v k^T, row j = v_j * k
    v[0, 0] = np.arange(D)
    o, S1 = oracle.delta(q, k, v, np.zeros((1, 1)), np.ones((1, 1)), np.zeros((1, D, D)), 0)
    assert np.array_equal(S1[0], np.outer(v[0, 0], k[0, 0]))


def test_decay_only_scales_state():
    q, k, v, g, _, S = _rand_case(12, 5, 1, 2, 8, g_scale=1.0)
    beta = np.zeros((5, 2))
    _, S1 = oracle.delta(q, k, v, g, beta, S, 0)
    for h in range(2):
        assert _rel(S1[h], S[h] * np.exp(np.sum(g[:, h]))) < 1e-14


def test_read_out_scale():
    """From zero state, beta=1, g=0, q=k unit: o = v (k.q) / sqrt(D) = v / sqrt(D)."""
    D = 4
    k = np.full((1, 1, D), 0.5)
    v = np.array([[[1.0, -2.0, 3.0, 0.5]]])
    o, _ = oracle.delta(k, k, v, np.zeros((1, 1)), np.ones((1, 1)), np.zeros((1, D, D)), 0)
    assert np.max(np.abs(o - v / 2.0)) < 1e-15


# ------------------------------------------------ O9: the chunk as an affine map
@pytest.mark.parametrize("chunk", [1, 7, 64, 145])
@pytest.mark.parametrize("g_scale", [0.02, 0.5, 8.0])
def test_affine_chunk_map_equals_recurrence(chunk, g_scale):
    T = 145
    q, k, v, g, beta, S = _rand_case(15, T, 2, 4, 16, g_scale=g_scale)
    for mp in (oracle.GROUPED, oracle.TILED):
        o, S1 = oracle.delta(q, k, v, g, beta, S, mp)
        oa, Sa = oracle.delta_affine(q, k, v, g, beta, S, mp, chunk)
        assert np.max(np.abs(oa - o)) < 1e-12 * max(1.0, np.max(np.abs(o)))
        assert np.max(np.abs(Sa - S1)) < 1e-12 * max(1.0, np.max(np.abs(S1)))


def test_affine_chunk_map_underflowing_decay():
    T = 70
    q, k, v, g, beta, S = _rand_case(16, T, 1, 2, 8)
    g = -np.random.default_rng(1).uniform(0, 50, size=(T, 2))
    o, S1 = oracle.delta(q, k, v, g, beta, S, oracle.GROUPED)
    oa, Sa = oracle.delta_affine(q, k, v, g, beta, S, oracle.GROUPED, 64)
    assert np.all(np.isfinite(oa)) and np.all(np.isfinite(Sa))
    assert np.max(np.abs(oa - o)) < 1e-12 and np.max(np.abs(Sa - S1)) < 1e-12


@pytest.mark.parametrize("mp", [oracle.GROUPED, oracle.TILED])
def test_chunk_factors_read_off_the_recurrence(mp):
    """Each factor, pinned to the token recurrence (O4) run on the chunk's
    tokens from chosen start states: S0 = 0 gives S_end = N and o = Y; S0 =
    e_a e_b^T (a one at value row a, key column b) adds row b of M to row a of
    S_end and column b of X to column a of o."""
    T, Hk, Hv, D = 9, 2, 4, 8
    q, k, v, g, beta, _ = _rand_case(17, T, Hk, Hv, D, g_scale=0.7)
    t0, L, h = 2, 6, 3
    M, N, X, Y = oracle.chunk_factors(q, k, v, g, beta, mp, h, t0, L)
    sl = slice(t0, t0 + L)

    def run(S0h):
        S = np.zeros((Hv, D, D))
        S[h] = S0h
        o, S1 = oracle.delta(q[sl], k[sl], v[sl], g[sl], beta[sl], S, mp)
        return o[:, h, :], S1[h]

    o0, s0 = run(np.zeros((D, D)))
    assert np.max(np.abs(s0 - N)) < 1e-12 and np.max(np.abs(o0 - Y)) < 1e-12
    for a, b in [(0, 0), (5, 2), (7, 7), (1, 6)]:
        E = np.zeros((D, D))
        E[a, b] = 1.0
        o1, s1 = run(E)
        assert np.max(np.abs((s1 - s0)[a] - M[b])) < 1e-12
        others = np.delete(s1 - s0, a, axis=0)
        assert np.max(np.abs(others)) < 1e-12  # no other row moves
        assert np.max(np.abs((o1 - o0)[:, a] - X[:, b])) < 1e-12
