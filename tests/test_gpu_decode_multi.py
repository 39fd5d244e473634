"""GPU checks of gdn_decode_multi (through the C ABI): T tokens per sequence
in one call, against T successive gdn_decode_step calls (bit for bit) and
against the fp64 oracle run over the same T tokens."""

import numpy as np
import pytest
import torch

import gdn_inputs as gi
import oracle
from tests.gpu_helpers import (DECODE_OUT_ABS, DECODE_STATE_REL, F64, assert_abs, assert_gated,
                               assert_state_rel, cuda)

pytestmark = pytest.mark.gpu


def _setup(shape, B, T, seed):
    g = gi.rng(seed)
    w = gi.layer_weights(g, shape)
    cs0 = gi.conv_state(g, shape, B, std=0.1)
    S0 = gi.delta_state(g, shape, B, std=0.05)
    steps = [gi.step_inputs(g, shape, B) for _ in range(T)]
    return w, cs0, S0, steps


def _stack(steps, name, B):
    """[T][B][...] step inputs -> [B][T][...] (token t of sequence b at [b][t])."""
    return torch.stack([getattr(s, name).reshape(B, -1) for s in steps], dim=1).contiguous()


def _run_multi(shape, w, cs0, S0, steps, core=True, norm=True):
    import gated_delta_net_causal_gb300 as gdn
    B, T = steps[0].mixed_qkv.shape[0], len(steps)
    Hv, D = shape.n_v_heads, shape.head_dim
    io = gi.DTYPES[shape.dtype]
    d = gdn.dims(shape.n_k_heads, Hv, D, shape.map, shape.decay, io)
    wd = {k: cuda(getattr(w, k)) for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
    cs, S = cuda(cs0), cuda(S0)
    core_out = torch.full((B, T, Hv, D), float("nan"), device="cuda") if core else None
    out = torch.full((B, T, Hv, D), float("nan"), device="cuda", dtype=io) if norm else None
    gdn.gdn_decode_multi(d, cuda(_stack(steps, "mixed_qkv", B)), cuda(_stack(steps, "a", B)),
                         cuda(_stack(steps, "b", B)), wd["decay_param"], wd["dt_bias"],
                         wd["conv_w"], cs, S, core_out=core_out,
                         z=cuda(_stack(steps, "z", B)).view(B, T, Hv, D) if norm else None,
                         norm_w=wd["norm_w"] if norm else None, out=out)
    torch.cuda.synchronize()
    return core_out, out, cs, S


def _run_steps(shape, w, cs0, S0, steps, core=True, norm=True):
    import gated_delta_net_causal_gb300 as gdn
    B, T = steps[0].mixed_qkv.shape[0], len(steps)
    Hv, D = shape.n_v_heads, shape.head_dim
    io = gi.DTYPES[shape.dtype]
    d = gdn.dims(shape.n_k_heads, Hv, D, shape.map, shape.decay, io)
    wd = {k: cuda(getattr(w, k)) for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
    cs, S = cuda(cs0), cuda(S0)
    cores, outs = [], []
    for x in steps:
        co = torch.full((B, Hv, D), float("nan"), device="cuda") if core else None
        o = torch.full((B, Hv, D), float("nan"), device="cuda", dtype=io) if norm else None
        gdn.gdn_decode_step(d, cuda(x.mixed_qkv), cuda(x.a), cuda(x.b), wd["decay_param"],
                            wd["dt_bias"], wd["conv_w"], cs, S, core_out=co,
                            z=cuda(x.z).view(B, Hv, D) if norm else None,
                            norm_w=wd["norm_w"] if norm else None, out=o)
        cores.append(co)
        outs.append(o)
    torch.cuda.synchronize()
    core_out = torch.stack(cores, dim=1) if core else None
    out = torch.stack(outs, dim=1) if norm else None
    return core_out, out, cs, S


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hk,hv,d", [(2, 4, 32), (2, 4, 64), (4, 8, 128), (2, 2, 128),
                                     (1, 8, 128), (2, 8, 64), (2, 4, 96)])
@pytest.mark.parametrize("T", [2, 5, 8])
def test_multi_equals_successive_steps_bitwise(dtype, hk, hv, d, T):
    mp, dec = (gi.TILED, gi.NEGATIVE_RATE) if (hk + T) % 2 else (gi.GROUPED, gi.LOG_RATE)
    shape = gi.Shape(hk, hv, d, map=mp, decay=dec, dtype=dtype)
    w, cs0, S0, steps = _setup(shape, 3, T, seed=5000 + 100 * hk + 10 * T + d)
    a = _run_multi(shape, w, cs0, S0, steps)
    b = _run_steps(shape, w, cs0, S0, steps)
    for name, x, y in zip(("core_out", "out", "conv_state", "state"), a, b):
        assert torch.equal(x, y), f"{shape} T={T}: {name} differs from {T} single steps"


def test_multi_core_only_and_norm_only():
    shape = gi.Shape(4, 8, 128, map=gi.TILED, decay=gi.LOG_RATE, dtype="bf16")
    w, cs0, S0, steps = _setup(shape, 2, 3, seed=5100)
    for core, norm in ((True, False), (False, True)):
        a = _run_multi(shape, w, cs0, S0, steps, core=core, norm=norm)
        b = _run_steps(shape, w, cs0, S0, steps, core=core, norm=norm)
        for x, y in zip(a, b):
            assert (x is None and y is None) or torch.equal(x, y)


def _oracle_multi(shape, w, cs0, S0, steps, seqs):
    """The oracle's decode over the T tokens of each sequence in `seqs`."""
    B, T = steps[0].mixed_qkv.shape[0], len(steps)
    cw, dp, dt, nw = F64(w.conv_w), F64(w.decay_param), F64(w.dt_bias), F64(w.norm_w)
    res = []
    for b in seqs:
        X = np.stack([F64(s.mixed_qkv)[b] for s in steps])
        A = np.stack([F64(s.a)[b] for s in steps])
        Bb = np.stack([F64(s.b)[b] for s in steps])
        Z = np.stack([F64(s.z)[b] for s in steps])
        res.append(oracle.segment(shape.n_k_heads, shape.n_v_heads, shape.head_dim, shape.map,
                                  shape.decay, X, A, Bb, Z, cw, dp, dt, nw, F64(cs0)[b],
                                  F64(S0)[b]))
    return res


@pytest.mark.parametrize("T", [2, 4, 8])
def test_multi_matches_the_oracle(T):
    shape = gi.Shape(4, 8, 128, map=gi.GROUPED, decay=gi.LOG_RATE, dtype="bf16")
    B = 3
    w, cs0, S0, steps = _setup(shape, B, T, seed=5200 + T)
    core_out, out, cs, S = _run_multi(shape, w, cs0, S0, steps)
    ref = _oracle_multi(shape, w, cs0, S0, steps, range(B))
    co, oy = F64(core_out.cpu()), F64(out.cpu())
    gS, gcs = F64(S.cpu()), F64(cs.cpu())
    for b, (rc, ry, rcs, rS) in enumerate(ref):
        tag = f"T={T} seq {b}"
        assert_abs(co[b], rc, DECODE_OUT_ABS, tag + " core")
        Z = np.stack([F64(s.z)[b] for s in steps])
        assert_gated(oy[b], ry, rc, Z, w.norm_w, shape.dtype, tag + " gated norm",
                     core_gpu=co[b])
        assert_state_rel(gS[b:b + 1], rS[None], DECODE_STATE_REL, tag + " state")
        assert np.array_equal(gcs[b], rcs), tag + " conv state (bitwise)"


def test_multi_full_size_four_tokens():
    """The batched-decode shape (B=64, Hk=16, Hv=32, D=128, Tiled,
    negative-rate, bf16) with 4 tokens per sequence: sampled sequences
    against the oracle, all of them against 4 single steps bit for bit."""
    shape = gi.Shape(16, 32, 128, map=gi.TILED, decay=gi.NEGATIVE_RATE, dtype="bf16")
    B, T = 64, 4
    w, cs0, S0, steps = _setup(shape, B, T, seed=5300)
    a = _run_multi(shape, w, cs0, S0, steps)
    b = _run_steps(shape, w, cs0, S0, steps)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    seqs = [0, 29, 63]
    ref = _oracle_multi(shape, w, cs0, S0, steps, seqs)
    co, gS = F64(a[0].cpu()), F64(a[3].cpu())
    for b_, (rc, ry, rcs, rS) in zip(seqs, ref):
        assert_abs(co[b_], rc, DECODE_OUT_ABS, f"seq {b_} core")
        assert_state_rel(gS[b_:b_ + 1], rS[None], DECODE_STATE_REL, f"seq {b_} state")


def test_multi_batch_zero_is_a_no_op():
    import gated_delta_net_causal_gb300 as gdn
    shape = gi.Shape(2, 4, 128, dtype="bf16")
    w, cs0, S0, steps = _setup(shape, 1, 2, seed=5400)
    d = gdn.dims(2, 4, 128, io_dtype=torch.bfloat16)
    S = cuda(S0)
    before = S.clone()
    C = gdn.gdn_qkv_features(d)
    empty = torch.empty((0, 2, C), device="cuda", dtype=torch.bfloat16)
    gdn.gdn_decode_multi(d, empty, torch.empty((0, 2, 4), device="cuda", dtype=torch.bfloat16),
                         torch.empty((0, 2, 4), device="cuda", dtype=torch.bfloat16),
                         cuda(w.decay_param), cuda(w.dt_bias), cuda(w.conv_w), cuda(cs0), S,
                         core_out=torch.empty((0, 2, 4, 128), device="cuda"))
    torch.cuda.synchronize()
    assert torch.equal(before, S)
