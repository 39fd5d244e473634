"""The seeded input recipe (gdn_inputs), checked on the CPU: values rounded
once to the storage dtype, and the workloads' shapes and laws as stated."""

import numpy as np
import pytest
import torch

import gdn_inputs as gi


def _neighbours(r: torch.Tensor):
    bits = r.view(torch.int16).to(torch.int32)
    lo = (bits - 1).to(torch.int16).view(r.dtype)
    hi = (bits + 1).to(torch.int16).view(r.dtype)
    return lo, hi


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rounding_is_once_to_nearest_even(dtype):
    rs = np.random.default_rng(3)
    x = rs.normal(size=20000) * rs.choice([1e-3, 1.0, 50.0], size=20000)
    # values a hair off a rounding midpoint of the 16-bit format, where a
    # conversion through float32 would round twice
    mant = 7 if dtype == "bf16" else 10
    base = 1.0 + rs.integers(0, 2 ** mant, size=2000) * 2.0 ** -mant
    mid = base + 2.0 ** -(mant + 1)
    x = np.concatenate([x, mid + 2.0 ** -40, mid - 2.0 ** -40, mid, -(mid + 2.0 ** -40)])
    r = gi.to_dtype(x, dtype)
    rv = gi.as_f64(r)
    lo, hi = _neighbours(r)
    err = np.abs(rv - x)
    for n in (gi.as_f64(lo), gi.as_f64(hi)):
        ok = np.isfinite(n) & (n != rv)
        assert np.all(err[ok] <= np.abs(n[ok] - x[ok])), "a neighbour is nearer"
    ties = np.zeros_like(err, dtype=bool)
    for n in (gi.as_f64(lo), gi.as_f64(hi)):
        ties |= np.isfinite(n) & (np.abs(n - x) == err) & (n != rv)
    even = (r.view(torch.int16).numpy() & 1) == 0
    assert np.all(even[ties]), "a tie not rounded to even"
    # the off-midpoint values go the way a single rounding sends them
    k = len(mid)
    up, down = rv[-4 * k:-3 * k], rv[-3 * k:-2 * k]
    assert np.all(up > base) and np.all(down == base)


def test_f32_is_plain_nearest_rounding():
    x = np.array([1.0 + 2.0 ** -24 + 2.0 ** -40, 0.1, -3.5])
    assert np.array_equal(gi.to_dtype(x, "f32").numpy(), x.astype(np.float32))


def test_batched_decode_recipe():
    wl = gi.workload_batched_decode(batch=64, sets=1)
    sh, w = wl["shape"], wl["weights"]
    assert (sh.n_k_heads, sh.n_v_heads, sh.head_dim, sh.map, sh.decay, sh.dtype) == (
        16, 32, 128, gi.TILED, gi.NEGATIVE_RATE, "bf16")
    assert tuple(wl["state"].shape) == (64, 32, 128, 128) and wl["state"].dtype == torch.float32
    assert abs(float(wl["state"].std()) - 0.02) < 0.0005
    assert tuple(wl["conv_state"].shape) == (64, 8192, 3)
    assert abs(float(wl["conv_state"].float().std()) - 0.1) < 0.002
    x = wl["steps"][0]
    assert tuple(x.mixed_qkv.shape) == (64, 8192) and abs(float(x.mixed_qkv.float().std()) - 1) < 0.02
    assert tuple(x.z.shape) == (64, 4096) and tuple(x.a.shape) == (64, 32)
    dp = w.decay_param.numpy()
    assert np.all((dp <= -1.0) & (dp >= -16.0))  # negative rate -U[1,16]
    assert np.all(np.abs(w.dt_bias.numpy()) <= 0.5)
    assert np.allclose(w.norm_w.numpy(), 0.82 + 0.013 * np.arange(128))


def test_single_layer_recipe():
    wl = gi.workload_single_layer_b1()
    w, x = wl["weights"], wl["inputs"]
    assert x.mixed_qkv.dtype == torch.float16 and tuple(x.mixed_qkv.shape) == (4, 8192)
    assert np.allclose(w.decay_param.numpy(), -1.7 + 0.07 * np.arange(32), atol=1e-6)
    assert np.allclose(w.dt_bias.numpy(), -0.25 + 0.04 * np.arange(32), atol=1e-6)
    # U(-0.04, 0.04) rounded to f16 may land half an f16 ulp past 0.04
    assert float(wl["conv_state"].float().abs().max()) <= 0.04 * (1 + 2.0 ** -11)
    assert float(wl["state"].abs().max()) <= 0.025 * (1 + 2.0 ** -24)


def test_multilayer_recipe_and_per_sequence_states():
    wl = gi.workload_multilayer_decode(layers=2, batch=4)
    sh = wl["shape"]
    assert (sh.n_v_heads, sh.qkv_features, sh.map, sh.decay) == (48, 10240, gi.GROUPED,
                                                                  gi.LOG_RATE)
    a_log = wl["weights"][0].decay_param.numpy()
    assert np.all((a_log >= 0.0) & (a_log <= np.log(16.0)))  # ln U[1,16]
    full = gi.multilayer_state(1, sh, 3, "cpu")
    assert torch.equal(gi.multilayer_state(1, sh, 3, "cpu", seqs=[2])[0], full[2])


def test_varlen_lengths_as_drawn():
    lengths = gi.varlen_lengths(gi.SEED_BASE + 5, 8, 512, 8192)
    assert lengths == [8110, 2965, 6963, 3562, 4169, 3929, 2191, 2593]
    assert sum(lengths) == 34482


def test_single_layer_sin_fill():
    """The deterministic fill: value i of each array is sin(i f) a, computed in
    float32 and rounded to f16 (the state stays float32)."""
    import math
    for decay in (gi.LOG_RATE, gi.NEGATIVE_RATE):
        wl = gi.workload_single_layer_sin(decay=decay)
        x, w = wl["inputs"], wl["weights"]
        assert tuple(x.mixed_qkv.shape) == (4, 8192) and x.mixed_qkv.dtype == torch.float16
        flat = x.mixed_qkv.reshape(-1)
        for i in (0, 1, 8193, 32767):
            ref = np.float16(np.float32(math.sin(np.float32(i) * np.float32(0.017))) *
                             np.float32(0.21))
            assert abs(float(flat[i]) - float(ref)) <= 2.0 ** -24 + abs(float(ref)) * 2.0 ** -10
        assert tuple(wl["state"].shape) == (1, 32, 128, 128) and wl["state"].dtype == torch.float32
        s1 = float(wl["state"].reshape(-1)[1])
        assert abs(s1 - math.sin(0.007) * 0.025) < 1e-8
        lr = -1.7 + 0.07 * np.arange(32)
        want = lr if decay == gi.LOG_RATE else -np.exp(lr)
        assert np.allclose(w.decay_param.numpy(), want, rtol=1e-6, atol=1e-6)
        assert tuple(wl["conv_state"].shape) == (1, 8192, 3)
