"""GPU parity of gdn_decode_step (through the C ABI) against the fp64 oracle."""

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests.gpu_helpers import (DECODE_OUT_ABS, DECODE_STATE_REL, DecodeRunner, F64, assert_abs,
                               assert_gated, assert_state_rel, cuda, decode_reference)

pytestmark = pytest.mark.gpu


def _check_steps(shape, batch, steps, seed, with_norm=True, core=True):
    g = gi.rng(seed)
    w = gi.layer_weights(g, shape)
    cs0 = gi.conv_state(g, shape, batch, std=0.1)
    S0 = gi.delta_state(g, shape, batch, std=0.05)
    run = DecodeRunner(shape, w, cs0, S0)
    cs, S = F64(cs0), F64(S0)
    for step in range(steps):
        x = gi.step_inputs(g, shape, batch)
        core_out, out = run.step(x, core=core, norm=with_norm)
        torch.cuda.synchronize()
        rc, ry, cs, S = decode_reference(shape, w, x, cs, S, with_norm=with_norm)
        tag = f"{shape} step {step}"
        if core:
            assert_abs(core_out, rc, DECODE_OUT_ABS, tag + " core")
        if with_norm:
            assert_gated(out, ry, rc, x.z, w.norm_w, shape.dtype, tag + " gated norm",
                         core_gpu=core_out)
        assert_state_rel(run.state, S, DECODE_STATE_REL, tag + " state")
        assert np.array_equal(F64(run.conv_state.cpu()), cs), tag + " conv state (bitwise)"
    assert run.gdn.gdn_device_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hk,hv,d", [(2, 4, 32), (2, 4, 64), (1, 2, 128), (4, 8, 128),
                                     (2, 2, 128), (1, 8, 128), (1, 16, 128), (2, 32, 64),
                                     (2, 4, 96), (1, 8, 96)])
@pytest.mark.parametrize("mp,dec", [(gi.GROUPED, gi.LOG_RATE), (gi.TILED, gi.NEGATIVE_RATE)])
def test_decode_small_shapes(dtype, hk, hv, d, mp, dec):
    shape = gi.Shape(hk, hv, d, map=mp, decay=dec, dtype=dtype)
    _check_steps(shape, batch=3, steps=3, seed=1000 + hk * 100 + hv * 10 + d + mp)


def test_decode_core_only_and_norm_only():
    shape = gi.Shape(2, 4, 128, map=gi.TILED, decay=gi.LOG_RATE, dtype="bf16")
    _check_steps(shape, batch=2, steps=2, seed=77, with_norm=False, core=True)
    _check_steps(shape, batch=2, steps=2, seed=78, with_norm=True, core=False)


def test_decode_batch_zero_is_a_no_op():
    shape = gi.Shape(2, 4, 128)
    g = gi.rng(3)
    w = gi.layer_weights(g, shape)
    run = DecodeRunner(shape, w, gi.conv_state(g, shape, 1), gi.delta_state(g, shape, 1))
    x = gi.step_inputs(g, shape, 0)
    before = run.state.clone()
    run.step(x)
    torch.cuda.synchronize()
    assert torch.equal(before, run.state)


def _permute_heads(shape, t, axis):
    """Reorder the V-head axis from grouped order to tiled order: grouped head
    kh*rep + r  ->  tiled head kh + r*Hk."""
    Hk, Hv = shape.n_k_heads, shape.n_v_heads
    rep = Hv // Hk
    perm = np.empty(Hv, dtype=np.int64)
    for kh in range(Hk):
        for r in range(rep):
            perm[kh + r * Hk] = kh * rep + r
    idx = torch.as_tensor(perm)
    return t.index_select(axis, idx), perm


def test_head_maps_are_a_pure_reindexing():
    """A grouped run and a tiled run on the same data, with every V-head
    indexed tensor permuted between the two orders, agree bit for bit."""
    Hk, Hv, D, B = 4, 8, 128, 3
    sg = gi.Shape(Hk, Hv, D, map=gi.GROUPED, decay=gi.LOG_RATE, dtype="bf16")
    st = gi.Shape(Hk, Hv, D, map=gi.TILED, decay=gi.LOG_RATE, dtype="bf16")
    g = gi.rng(91)
    w = gi.layer_weights(g, sg)
    x = gi.step_inputs(g, sg, B)
    cs = gi.conv_state(g, sg, B)
    S = gi.delta_state(g, sg, B)
    C, qk = sg.qkv_features, 2 * Hk * D
    # tiled copies: permute v channels, conv rows of v, gates, params, state, z
    def perm_v_channels(t, axis):
        head = t.narrow(axis, qk, Hv * D)
        shp = list(head.shape)
        shp[axis:axis + 1] = [Hv, D]
        ph, _ = _permute_heads(sg, head.reshape(shp), axis)
        return torch.cat([t.narrow(axis, 0, qk), ph.reshape(head.shape)], axis)
    wt = gi.Weights(conv_w=perm_v_channels(w.conv_w, 0),
                    decay_param=_permute_heads(sg, w.decay_param, 0)[0],
                    dt_bias=_permute_heads(sg, w.dt_bias, 0)[0], norm_w=w.norm_w)
    xt = gi.StepInputs(mixed_qkv=perm_v_channels(x.mixed_qkv, 1),
                       a=_permute_heads(sg, x.a, 1)[0], b=_permute_heads(sg, x.b, 1)[0],
                       z=_permute_heads(sg, x.z.view(B, Hv, D), 1)[0].reshape(B, Hv * D))
    cst = perm_v_channels(cs, 1)
    Sg = _permute_heads(sg, S, 1)[0]
    rg = DecodeRunner(sg, w, cs, S)
    rt = DecodeRunner(st, wt, cst, Sg)
    og, yg = rg.step(x)
    ot, yt = rt.step(xt)
    torch.cuda.synchronize()
    assert torch.equal(_permute_heads(sg, og.cpu(), 1)[0], ot.cpu())
    assert torch.equal(_permute_heads(sg, yg.cpu(), 1)[0], yt.cpu())
    assert torch.equal(_permute_heads(sg, rg.state.cpu(), 1)[0], rt.state.cpu())
    assert torch.equal(perm_v_channels(rg.conv_state.cpu(), 1), rt.conv_state.cpu())


def test_decode_tagged_heads_read_the_mapped_k_head():
    """With zero conv state, conv weight taps (0,0,0,w3) and inputs chosen per
    K head, every V head's output depends only on which K head it read; the
    outputs must match the oracle's exactly-indexed result for both maps."""
    for mp in (gi.GROUPED, gi.TILED):
        shape = gi.Shape(4, 8, 128, map=mp, decay=gi.LOG_RATE, dtype="f32")
        g = gi.rng(5)
        w = gi.layer_weights(g, shape)
        C = shape.qkv_features
        cw = torch.zeros(C, 4)
        cw[:, 3] = 1.0
        w.conv_w = cw
        x = gi.step_inputs(g, shape, 1)
        xm = torch.zeros_like(x.mixed_qkv)
        D, Hk = 128, 4
        for kh in range(Hk):
            xm[0, kh * D + kh] = 3.0  # q of K head kh: one-hot at column kh
            xm[0, Hk * D + kh * D + kh] = 3.0  # k likewise
        xm[0, 2 * Hk * D:] = x.mixed_qkv[0, 2 * Hk * D:]
        x.mixed_qkv = xm
        cs = torch.zeros(1, C, 3)
        S = gi.delta_state(g, shape, 1)
        run = DecodeRunner(shape, w, cs, S)
        core, _ = run.step(x, norm=False)
        torch.cuda.synchronize()
        rc, _, _, _ = decode_reference(shape, w, x, F64(cs), F64(S), with_norm=False)
        assert_abs(core, rc, DECODE_OUT_ABS, f"tagged heads map={mp}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_decode_reads_and_writes_pinned_host_memory(dtype):
    """Activations, z and both outputs in mapped pinned host memory (read and
    written by the kernel over the host link): the same bits as the call on
    device copies, for several steps in a row."""
    import gated_delta_net_causal_gb300 as gdn
    shape = gi.Shape(2, 4, 128, map=gi.TILED, decay=gi.NEGATIVE_RATE, dtype=dtype)
    g = gi.rng(91)
    w = gi.layer_weights(g, shape)
    cs0, S0 = gi.conv_state(g, shape, 5), gi.delta_state(g, shape, 5)
    dev = DecodeRunner(shape, w, cs0, S0)
    host = DecodeRunner(shape, w, cs0, S0)
    io = gi.DTYPES[dtype]
    for step in range(3):
        x = gi.step_inputs(g, shape, 5)
        B, Hv, D = 5, shape.n_v_heads, shape.head_dim
        pin = {k: getattr(x, k).contiguous().pin_memory() for k in ("mixed_qkv", "a", "b", "z")}
        assert gdn.gdn_host_pointer(pin["a"]) != 0
        core_h = torch.full((B, Hv, D), float("nan")).pin_memory()
        out_h = torch.full((B, Hv, D), float("nan"), dtype=io).pin_memory()
        gdn.gdn_decode_step(host.d, pin["mixed_qkv"], pin["a"], pin["b"], host.w["decay_param"],
                            host.w["dt_bias"], host.w["conv_w"], host.conv_state, host.state,
                            core_out=core_h, z=pin["z"].view(B, Hv, D), norm_w=host.w["norm_w"],
                            out=out_h)
        core_d, out_d = dev.step(x)
        torch.cuda.synchronize()
        assert torch.equal(core_h, core_d.cpu()), f"step {step}: core output"
        assert torch.equal(out_h, out_d.cpu()), f"step {step}: gated output"
        assert torch.equal(host.state, dev.state) and torch.equal(host.conv_state, dev.conv_state)


# With decays near 1 the state keeps every step's rounding, so errors of
# successive steps add: ten times the single-step state bound after 32 steps
# (the fp32 rounding of 32 kept steps is a few 1e-6 of the state's largest
# magnitude; a dropped decay moves it by about 3e-2 over those steps, a sign
# error by its own size).
LONG_STATE_REL = 10 * DECODE_STATE_REL


@pytest.mark.parametrize("mp,dec", [(gi.GROUPED, gi.LOG_RATE), (gi.TILED, gi.NEGATIVE_RATE)])
def test_decode_long_memory_many_steps(mp, dec):
    """32 consecutive steps with decay rates of about 1e-3 per token
    (A_log = ln U[5e-4, 2e-3], so the state carries across all of them):
    every step's outputs against the oracle at the decode bounds, the state
    within LONG_STATE_REL; then the same 32 tokens as four 8-token
    gdn_decode_multi calls from the same start, against the same oracle."""
    import gated_delta_net_causal_gb300 as gdn
    shape = gi.Shape(2, 4, 128, map=mp, decay=dec, dtype="bf16")
    B, steps = 3, 32
    g = gi.rng(777)
    a_log = np.log(g.uniform(5e-4, 2e-3, size=shape.n_v_heads))
    w = gi.layer_weights(g, shape, a_log=a_log)
    cs0 = gi.conv_state(g, shape, B, std=0.1)
    S0 = gi.delta_state(g, shape, B, std=0.05)
    xs = [gi.step_inputs(g, shape, B) for _ in range(steps)]
    g_tok, _ = oracle.gates(F64(xs[0].a), F64(xs[0].b), F64(w.decay_param), F64(w.dt_bias), dec)
    assert float(np.median(g_tok)) > -5e-3, "the case must have long memory"

    run = DecodeRunner(shape, w, cs0, S0)
    cs, S = F64(cs0), F64(S0)
    refs = []
    for step, x in enumerate(xs):
        core_out, out = run.step(x)
        torch.cuda.synchronize()
        rc, ry, cs, S = decode_reference(shape, w, x, cs, S)
        refs.append(rc)
        tag = f"{shape} long-memory step {step}"
        assert_abs(core_out, rc, DECODE_OUT_ABS, tag + " core")
        assert_gated(out, ry, rc, x.z, w.norm_w, shape.dtype, tag + " gated norm",
                     core_gpu=core_out)
        assert_state_rel(run.state, S, LONG_STATE_REL, tag + " state")
        assert np.array_equal(F64(run.conv_state.cpu()), cs), tag + " conv state (bitwise)"

    multi = DecodeRunner(shape, w, cs0, S0)
    Hv, D = shape.n_v_heads, shape.head_dim
    for c in range(steps // 8):
        blk = xs[8 * c:8 * c + 8]

        def stack(name):
            return cuda(torch.stack([getattr(s, name).reshape(B, -1) for s in blk], dim=1))
        core = torch.full((B, 8, Hv, D), float("nan"), device="cuda")
        gdn.gdn_decode_multi(multi.d, stack("mixed_qkv"), stack("a"), stack("b"),
                             multi.w["decay_param"], multi.w["dt_bias"], multi.w["conv_w"],
                             multi.conv_state, multi.state, core_out=core)
        torch.cuda.synchronize()
        for t in range(8):
            assert_abs(core[:, t], refs[8 * c + t], DECODE_OUT_ABS, f"multi call {c} token {t}")
    assert_state_rel(multi.state, S, LONG_STATE_REL, "multi-token long-memory state")
    assert np.array_equal(F64(multi.conv_state.cpu()), cs), "multi-token conv state (bitwise)"
    assert gdn.gdn_device_error() == 0
