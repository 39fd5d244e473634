"""Pins for the fp64 oracle: the pages' printed values, closed forms and
library routines that the oracle's own code does not use."""

import json
import math
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN

MAPS = {"tiled": oracle.TILED, "grouped": oracle.GROUPED}


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- printed values

def test_scalar_worked_example():
    gd = _golden("scalar_recurrence.json")
    q = np.array(gd["q"]).reshape(1, 1, 1)
    k = np.array(gd["k"]).reshape(1, 1, 1)
    v = np.array(gd["v"]).reshape(1, 1, 1)
    g = np.array(gd["g"]).reshape(1, 1)
    beta = np.array(gd["beta"]).reshape(1, 1)
    S = np.array(gd["state_in"]).reshape(1, 1, 1)
    for fn in (oracle.delta, oracle.delta_chunked, oracle.delta_bruteforce):
        o, S1 = fn(q, k, v, g, beta, S, MAPS[gd["map"]])
        assert abs(S1.ravel()[0] - gd["expected_state"][0]) < gd["tolerance"]
        assert abs(o.ravel()[0] - gd["expected_out"][0]) < gd["tolerance"]


def test_head_map_indices():
    gd = _golden("head_maps.json")
    for c in gd["k_head_cases"]:
        assert oracle.k_head(MAPS[c["map"]], c["v_head"], c["n_k"], c["n_v"]) == c["k_head"]


@pytest.mark.parametrize("name", ["tiled", "grouped"])
def test_head_map_step_example(name):
    st = _golden("head_maps.json")["step"]
    Hk, Hv, D = st["n_k_heads"], st["n_v_heads"], st["head_dim"]
    q = np.array(st["q"]).reshape(1, Hk, D)
    k = np.array(st["k"]).reshape(1, Hk, D)
    v = np.array(st["v"]).reshape(1, Hv, D)
    g = np.array(st["g"]).reshape(1, Hv)
    beta = np.array(st["beta"]).reshape(1, Hv)
    S = np.array(st["state_in"]).reshape(Hv, D, D)
    for fn in (oracle.delta, oracle.delta_chunked, oracle.delta_bruteforce):
        o, _ = fn(q, k, v, g, beta, S, MAPS[name])
        assert o.ravel().tolist() == st[f"expected_out_{name}"]


def test_l2_normalize_example():
    gd = _golden("l2_normalize.json")
    for c in gd["cases"]:
        x = np.array([c["x"]])
        y = oracle.l2norm(x, gd["eps"], clamped=True)
        assert np.max(np.abs(y - np.array([c["expected"]]))) <= c["tolerance"]
        # the (sum + eps)^(-1/2) form agrees within the same tolerance here
        y2 = oracle.l2norm(x, gd["eps"], clamped=False)
        assert np.max(np.abs(y2 - np.array([c["expected"]]))) <= max(c["tolerance"], 1e-12)


def test_l2_normalize_many_rows_against_numpy():
    """O2 over a (5, 3, 7) array, rows of different scales, against
    numpy.linalg.norm row by row: a row-indexing or stride mistake in either
    form fails here (the page's example has a single row)."""
    rng = np.random.default_rng(20261203)
    x = rng.normal(size=(5, 3, 7)) * rng.uniform(0.01, 100.0, size=(5, 3, 1))
    x[2, 1] = 0.0  # an all-zero row
    n = np.linalg.norm(x, axis=-1, keepdims=True)
    eps = 1e-6
    assert np.allclose(oracle.l2norm(x, eps, clamped=True), x / np.maximum(n, eps), rtol=1e-14, atol=0)
    assert np.allclose(oracle.l2norm(x, eps, clamped=False), x / np.sqrt(n * n + eps), rtol=1e-14, atol=0)
    # every nonzero row has unit norm up to the eps term
    y = oracle.l2norm(x, 0.0, clamped=True)
    norms = np.linalg.norm(y, axis=-1)
    assert np.allclose(np.delete(norms.ravel(), 2 * 3 + 1), 1.0, rtol=1e-14)


# -------------------------------------------------------------- closed forms

def test_sigmoid_softplus_silu_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.softplus(0.0) - math.log(2.0)) < 1e-15
    assert oracle.silu(0.0) == 0.0
    xs = np.concatenate([np.linspace(-40, 40, 161), [-1e-3, 1e-3, 19.999, 20.001, -20.001]])
    for x in xs:
        s, sm = oracle.sigmoid(x), oracle.sigmoid(-x)
        assert abs(s + sm - 1.0) < 1e-15
        # numpy's logaddexp(0, x) = log(1 + e^x) is an independent routine
        ref = float(np.logaddexp(0.0, x))
        sp = oracle.softplus(x)
        # the piecewise cut-offs at +-20 change the value by < 2.1e-9 relative
        assert abs(sp - ref) <= 2.1e-9 * max(abs(ref), 1e-300), (x, sp, ref)
        if abs(x) < 20:
            assert abs(oracle.softplus(x) - oracle.softplus(-x) - x) < 1e-12
        assert abs(oracle.silu(x) - x / (1.0 + math.exp(-x))) <= 1e-15 * max(1.0, abs(x))


def test_gates_against_library_forms():
    rng = np.random.default_rng(5)
    T, Hv = 3, 6
    a, b = rng.normal(size=(T, Hv)), rng.normal(size=(T, Hv)) * 3
    A_log = np.log(rng.uniform(1, 16, Hv))
    dt = rng.uniform(-0.5, 0.5, Hv)
    g, beta = oracle.gates(a, b, A_log, dt, oracle.LOG_RATE)
    ref_g = -np.exp(A_log)[None, :] * np.logaddexp(0.0, a + dt[None, :])
    ref_b = 0.5 * (1.0 + np.tanh(0.5 * b))  # logistic via tanh identity
    assert np.max(np.abs(g - ref_g) / np.abs(ref_g)) < 1e-13
    assert np.max(np.abs(beta - ref_b)) < 1e-15
    # negative-rate form with the same rate gives the same g
    g2, beta2 = oracle.gates(a, b, -np.exp(A_log), dt, oracle.NEGATIVE_RATE)
    assert np.max(np.abs(g2 - g) / np.abs(g)) < 1e-15
    assert np.array_equal(beta2, beta)


def _conv_numpy(x, w, state):
    """Per channel: history then inputs, correlated with the 4 taps (numpy's
    convolve with the taps reversed), then SiLU; the new state is the last
    three entries of history+inputs."""
    T, C = x.shape
    y = np.zeros((T, C))
    new = np.zeros((C, 3))
    for c in range(C):
        seq = np.concatenate([state[c], x[:, c]])
        if T > 0:
            lin = np.convolve(seq, w[c][::-1], mode="valid")
            y[:, c] = lin / (1.0 + np.exp(-lin))
        new[c] = seq[-3:]
    return y, new


@pytest.mark.parametrize("T", [0, 1, 2, 3, 4, 9])
def test_conv_matches_numpy_convolve(T):
    rng = np.random.default_rng(100 + T)
    C = 6
    x, w, st = rng.normal(size=(T, C)), rng.normal(size=(C, 4)), rng.normal(size=(C, 3))
    y, new = oracle.conv(x, w, st)
    yr, newr = _conv_numpy(x, w, st)
    assert y.shape == (T, C)
    assert np.max(np.abs(y - yr), initial=0.0) < 1e-13
    assert np.array_equal(new, newr)  # the state is a copy of raw values


def test_conv_zero_input_and_varlen_independence():
    rng = np.random.default_rng(7)
    C = 5
    y, new = oracle.conv(np.zeros((4, C)), rng.normal(size=(C, 4)), np.zeros((C, 3)))
    assert not y.any() and not new.any()
    lens = [3, 0, 5, 1]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.normal(size=(cu[-1], C))
    w = rng.normal(size=(C, 4))
    sts = rng.normal(size=(len(lens), C, 3))
    y, new = oracle.conv_varlen(x, w, sts, cu)
    for n in range(len(lens)):
        yn, sn = _conv_numpy(x[cu[n]:cu[n + 1]], w, sts[n])
        assert np.max(np.abs(y[cu[n]:cu[n + 1]] - yn), initial=0.0) < 1e-13
        assert np.array_equal(new[n], sn)


def test_gated_rmsnorm_constant_row_closed_form():
    D = 16
    rng = np.random.default_rng(3)
    w = rng.uniform(0.5, 1.5, D)
    z = rng.normal(size=(1, D))
    eps = 1e-6
    for c in (0.37, -2.5, 1e-4):
        o = np.full((1, D), c)
        y = oracle.gated_rmsnorm(o, z, w, eps)
        silu = z / (1.0 + np.exp(-z))
        ref = np.sign(c) * w * silu / np.sqrt(1.0 + eps / (c * c))
        assert np.max(np.abs(y - ref)) < 1e-14


def test_gated_rmsnorm_scale_invariance_and_zero_gate():
    rng = np.random.default_rng(4)
    D = 32
    o = rng.normal(size=(3, D))
    z = rng.normal(size=(3, D))
    w = rng.normal(size=D)
    y1 = oracle.gated_rmsnorm(o, z, w, 0.0)
    y2 = oracle.gated_rmsnorm(o * 7.25, z, w, 0.0)
    assert np.max(np.abs(y1 - y2)) < 1e-13
    # unit RMS row, eps 0: y = o * w * silu(z); with z = 0 the gate closes
    assert not oracle.gated_rmsnorm(o, np.zeros_like(z), w, 1e-6).any()
    # rows of unit RMS pass through scaled by w * silu(z)
    u = o / np.sqrt(np.mean(o * o, axis=1, keepdims=True))
    y3 = oracle.gated_rmsnorm(u, z, w, 0.0)
    assert np.max(np.abs(y3 - u * w * (z / (1 + np.exp(-z))))) < 1e-13


def test_segment_composes_the_steps():
    """O6 equals O1 -> split -> O2 -> O3 -> O4 -> O5 called one by one."""
    rng = np.random.default_rng(11)
    Hk, Hv, D, T = 2, 4, 8, 5
    C = 2 * Hk * D + Hv * D
    x = rng.normal(size=(T, C))
    a, b = rng.normal(size=(T, Hv)), rng.normal(size=(T, Hv))
    z = rng.normal(size=(T, Hv, D))
    w = rng.normal(size=(C, 4)) * 0.4
    A_log, dt = np.log(rng.uniform(1, 4, Hv)), rng.uniform(-0.5, 0.5, Hv)
    nw = rng.uniform(0.8, 1.2, D)
    cs, S = rng.normal(size=(C, 3)), rng.normal(size=(Hv, D, D)) * 0.1
    core, y, cs1, S1 = oracle.segment(Hk, Hv, D, oracle.TILED, oracle.LOG_RATE, x, a, b, z, w,
                                      A_log, dt, nw, cs, S)
    yc, csr = oracle.conv(x, w, cs)
    q = oracle.l2norm(yc[:, :Hk * D].reshape(T, Hk, D))
    k = oracle.l2norm(yc[:, Hk * D:2 * Hk * D].reshape(T, Hk, D))
    v = yc[:, 2 * Hk * D:].reshape(T, Hv, D)
    g, beta = oracle.gates(a, b, A_log, dt, oracle.LOG_RATE)
    o, Sr = oracle.delta(q, k, v, g, beta, S, oracle.TILED)
    assert np.array_equal(cs1, csr)
    assert np.array_equal(core, o)
    assert np.array_equal(S1, Sr)
    assert np.array_equal(y, oracle.gated_rmsnorm(o, z, nw))


# ------------------------------------------------------------- decode layer

def test_round_bf16_against_torch_and_ties():
    """round_bf16 agrees with torch's own float -> bfloat16 conversion (a
    library routine) on random values of every scale, and rounds the exact
    ties to even."""
    import torch
    rng = np.random.default_rng(7)
    x = rng.normal(size=4000) * np.exp(rng.uniform(-30, 30, size=4000))
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oracle.round_bf16(x), ref)
    one_ulp = 2.0 ** -7
    assert oracle.round_bf16(1.0 + one_ulp / 2) == 1.0                   # tie, even below
    assert oracle.round_bf16(1.0 + 1.5 * one_ulp) == 1.0 + 2 * one_ulp   # tie, even above
    assert oracle.round_bf16(1.0 + 0.75 * one_ulp) == 1.0 + one_ulp


def test_linear_against_a_brute_force_sum():
    """linear = an fsum triple loop (bias added, one rounding) on small
    random shapes; without rounding it is the exact fp64 sum of products."""
    rng = np.random.default_rng(11)
    x = oracle.round_bf16(rng.normal(size=(3, 20)))
    w = oracle.round_bf16(rng.normal(size=(7, 20)))
    bias = rng.normal(size=7)
    exact = np.array([[math.fsum([x[m, k] * w[n, k] for k in range(20)] + [bias[n]]) for n in range(7)]
                      for m in range(3)])
    assert np.allclose(oracle.linear(x, w, bias, round_out=False), exact, rtol=1e-15, atol=1e-15)
    assert np.array_equal(oracle.linear(x, w, bias), oracle.round_bf16(exact))


def test_decode_layer_with_selection_weights_is_the_segment():
    """With input weights that copy given bf16 values of qkv, z, b, a out of
    the input (one 1 per row) and an output projection that copies the gated
    core output, the layer is O6 (already pinned) plus the bf16 roundings."""
    Hk, Hv, D = 2, 4, 32
    C, vw = (2 * Hk + Hv) * D, Hv * D
    n = C + vw + 2 * Hv
    hidden = n
    rng = np.random.default_rng(5)
    B = 2
    x = oracle.round_bf16(rng.normal(size=(B, hidden)) * 0.5)
    w_in = np.eye(n)  # row r picks input feature r
    w_out = np.zeros((vw, vw))
    w_out[np.arange(vw), np.arange(vw)] = 1.0
    conv_w = rng.normal(size=(C, 4)) * 0.3
    dp, dt = rng.normal(size=Hv) * 0.2 - 1.0, rng.normal(size=Hv) * 0.1
    nw = rng.normal(size=D) * 0.1 + 1.0
    cs0 = rng.normal(size=(B, C, 3)) * 0.1
    S0 = rng.normal(size=(B, Hv, D, D)) * 0.02
    out, cs, S, yc = oracle.decode_layer(Hk, Hv, D, oracle.GROUPED, oracle.LOG_RATE, x, w_in, None, w_out,
                                         None, conv_w, dp, dt, nw, cs0, S0)
    for b in range(B):
        core, y, cs_b, S_b = oracle.segment(Hk, Hv, D, oracle.GROUPED, oracle.LOG_RATE, x[b:b + 1, :C],
                                            x[b:b + 1, C + vw + Hv:C + vw + 2 * Hv],
                                            x[b:b + 1, C + vw:C + vw + Hv], x[b:b + 1, C:C + vw], conv_w, dp,
                                            dt, nw, cs0[b], S0[b])
        assert np.array_equal(yc[b], oracle.round_bf16(y[0]))
        assert np.array_equal(out[b], oracle.round_bf16(yc[b].reshape(-1)))
        assert np.array_equal(cs[b], cs_b) and np.array_equal(S[b], S_b)
