"""The five synthetic workloads at their full sizes on the GPU, in the launch
configuration the benchmark times, with the oracle recomputing sampled
sequences, heads and layers (each independent of the rest)."""

import numpy as np
import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
import gdn_inputs as gi
import oracle
from tests.gpu_helpers import (CHUNK_OUT_ABS, CHUNK_STATE_ABS, DECODE_OUT_ABS, DECODE_STATE_REL,
                               DecodeRunner, F64, assert_abs, assert_gated, assert_lowp,
                               assert_state_rel, cuda, decode_reference, parallel_map)

pytestmark = pytest.mark.gpu


# ------------------------------------------------------------ single layer, B=1

@pytest.mark.parametrize("source", ["seeded", "sin_fill"])
@pytest.mark.parametrize("mp,dec", [(gi.GROUPED, gi.LOG_RATE), (gi.TILED, gi.NEGATIVE_RATE)])
def test_single_layer_b1_four_tokens_and_split(mp, dec, source):
    """(i) four tokens decoded one at a time; (ii) the first three as one
    segment (conv update + chunked prefill, one partial chunk) then one decode
    step. (i) at the decode bounds, (ii) at the chunk bounds, against the
    oracle and against each other. On the seeded inputs and, as a
    cross-check, on the Metal conformance test's deterministic sin fill."""
    if source == "seeded":
        wl = gi.workload_single_layer_b1(dtype="f16", map=mp, decay=dec)
    else:
        wl = gi.workload_single_layer_sin(map=mp, decay=dec)
    shape, w, x = wl["shape"], wl["weights"], wl["inputs"]
    D, Hv, Hk, C = 128, 32, 16, shape.qkv_features
    # oracle over the whole 4-token segment
    rc, ry, rcs, rS = oracle.segment(Hk, Hv, D, mp, dec, F64(x.mixed_qkv), F64(x.a), F64(x.b),
                                     F64(x.z), F64(w.conv_w), F64(w.decay_param),
                                     F64(w.dt_bias), F64(w.norm_w), F64(wl["conv_state"])[0],
                                     F64(wl["state"])[0])
    # (i)
    run = DecodeRunner(shape, w, wl["conv_state"], wl["state"])
    cores, outs = [], []
    for t in range(4):
        xt = gi.StepInputs(x.mixed_qkv[t:t + 1], x.a[t:t + 1], x.b[t:t + 1], x.z[t:t + 1])
        c, o = run.step(xt)
        cores.append(c.cpu())
        outs.append(o.cpu())
    torch.cuda.synchronize()
    full_core = torch.cat(cores)
    full_out = torch.cat(outs)
    assert (full_out.abs() > 1e-4).any()
    assert_abs(full_core, rc, DECODE_OUT_ABS, "4 x decode output")
    assert_gated(full_out, ry, rc, x.z, w.norm_w, "f16", "4 x decode gated output",
                 core_gpu=full_core)
    assert_state_rel(run.state.cpu(), rS[None], DECODE_STATE_REL, "4 x decode state")
    assert np.array_equal(F64(run.conv_state.cpu())[0], rcs)

    # (ii) 3-token segment then 1 decode
    d = gdn.dims(Hk, Hv, D, map=mp, decay=dec, io_dtype=torch.float16)
    cs2, S2 = cuda(wl["conv_state"]), cuda(wl["state"])
    xs = cuda(x.mixed_qkv[:3])
    y = torch.empty_like(xs)
    cu = cuda(gi.cu_seqlens([3]))
    gdn.gdn_conv_update(d, cu, xs, cuda(w.conv_w), cs2, y)
    qk = Hk * D
    core3 = torch.empty((3, Hv, D), device="cuda")
    out3 = torch.empty((3, Hv, D), device="cuda", dtype=torch.float16)
    gdn.gdn_prefill_chunked(d, cu, y[:, :qk], y[:, qk:2 * qk], y[:, 2 * qk:], cuda(x.a[:3]),
                            cuda(x.b[:3]), cuda(w.decay_param), cuda(w.dt_bias), S2,
                            core_out=core3, z=cuda(x.z[:3]).view(3, Hv, D),
                            norm_w=cuda(w.norm_w), out=out3)
    run2 = DecodeRunner(shape, w, wl["conv_state"], wl["state"])
    run2.conv_state, run2.state = cs2, S2
    c4, o4 = run2.step(gi.StepInputs(x.mixed_qkv[3:], x.a[3:], x.b[3:], x.z[3:]))
    torch.cuda.synchronize()
    split_core = torch.cat([core3.cpu(), c4.cpu()])
    split_out = torch.cat([out3.cpu(), o4.cpu()])
    assert_abs(split_core, rc, CHUNK_OUT_ABS, "3+1 output vs oracle")
    assert_abs(split_core, F64(full_core), CHUNK_OUT_ABS, "3+1 output vs 4 x decode")
    assert_abs(S2.cpu()[0], rS, CHUNK_STATE_ABS, "3+1 state vs oracle")
    assert np.array_equal(F64(cs2.cpu())[0], rcs), "3+1 conv state"
    # gated outputs of the split run, with the chunk bound carried through the norm
    assert_gated(split_out, ry, rc, x.z, w.norm_w, "f16", "3+1 gated output",
                 core_gpu=split_core, eps_o=CHUNK_OUT_ABS)


# ----------------------------------------------------------- batched decode, B=64

def test_batched_decode_b64_sampled_sequences():
    """B=64, 16 consecutive steps (the 16 input sets) on the GPU; sequences
    0, 31, 63 checked after steps 1, 2 and 16."""
    wl = gi.workload_batched_decode(batch=64, sets=16)
    shape, w = wl["shape"], wl["weights"]
    run = DecodeRunner(shape, w, wl["conv_state"], wl["state"])
    seqs = [0, 31, 63]
    cs = F64(wl["conv_state"])[seqs]
    S = F64(wl["state"])[seqs]
    for step in range(16):
        x = wl["steps"][step]
        core, out = run.step(x)
        rc, ry, cs, S = decode_reference(shape, w, x, cs, S, seqs=seqs)
        if step in (0, 1, 15):
            torch.cuda.synchronize()
            tag = f"B=64 step {step + 1}"
            assert_abs(core.cpu()[seqs], rc, DECODE_OUT_ABS, tag + " output")
            assert_gated(out.cpu()[seqs], ry, rc, F64(x.z)[seqs], w.norm_w, "bf16",
                         tag + " gated output", core_gpu=core.cpu()[seqs])
            assert_state_rel(run.state.cpu()[seqs], S, DECODE_STATE_REL, tag + " state")
            assert np.array_equal(F64(run.conv_state.cpu())[seqs], cs), tag + " conv state"
    assert gdn.gdn_device_error() == 0


# ------------------------------------------------------ 48 layers x B=128 decode

def test_multilayer_decode_48x128_sampled():
    """48 layers x B=128, Hv=48 (18 GiB of fp32 state) run back to back on one
    stream; sequences {0, 77, 127} x layers {0, 23, 47} checked."""
    L, B = 48, 128
    wl = gi.workload_multilayer_decode(layers=L, batch=B)
    shape = wl["shape"]
    seqs, layers = [0, 77, 127], [0, 23, 47]
    d = gdn.dims(16, 48, 128, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    states, init = [], {}
    for l in range(L):
        gen = torch.Generator(device="cuda").manual_seed(gi.SEED_BASE + 3 + 1000 * (l + 1))
        s = torch.randn((B, 48, 128, 128), device="cuda", generator=gen) * 0.02
        states.append(s)
        if l in layers:
            init[l] = F64(s[seqs].cpu())
    convs = [cuda(c) for c in wl["conv_states"]]
    outs = []
    for l in range(L):
        w, x = wl["weights"][l], wl["inputs"][l]
        out = torch.empty((B, 48, 128), device="cuda", dtype=torch.bfloat16)
        core = torch.empty((B, 48, 128), device="cuda")
        gdn.gdn_decode_step(d, cuda(x.mixed_qkv), cuda(x.a), cuda(x.b), cuda(w.decay_param),
                            cuda(w.dt_bias), cuda(w.conv_w), convs[l], states[l], core_out=core,
                            z=cuda(x.z).view(B, 48, 128), norm_w=cuda(w.norm_w), out=out)
        outs.append((core, out))
    torch.cuda.synchronize()
    for l in layers:
        w, x = wl["weights"][l], wl["inputs"][l]
        rc, ry, rcs, rS = decode_reference(shape, w, x, F64(wl["conv_states"][l])[seqs],
                                           init[l], seqs=seqs)
        tag = f"layer {l}"
        assert_abs(outs[l][0].cpu()[seqs], rc, DECODE_OUT_ABS, tag + " output")
        assert_gated(outs[l][1].cpu()[seqs], ry, rc, F64(x.z)[seqs], w.norm_w, "bf16",
                     tag + " gated output", core_gpu=outs[l][0].cpu()[seqs])
        assert_state_rel(states[l][seqs].cpu(), rS, DECODE_STATE_REL, tag + " state")
        assert np.array_equal(F64(convs[l].cpu())[seqs], rcs), tag + " conv state"
    del states


# ------------------------------------------- varlen prefill then decode, ~32k tokens

def _head_channels(shape, h):
    Hk, Hv, D = shape.n_k_heads, shape.n_v_heads, shape.head_dim
    kh = oracle.k_head(shape.map, h, Hk, Hv)
    qk = Hk * D
    return np.concatenate([np.arange(kh * D, (kh + 1) * D), qk + np.arange(kh * D, (kh + 1) * D),
                           2 * qk + np.arange(h * D, (h + 1) * D)])


def test_varlen_prefill_then_decode():
    """8 sequences (lengths U[512,8192] as drawn) packed by cu_seqlens, each
    resuming from a prior state and conv state: conv update, chunked prefill
    with the fused norm, then 16 batched decode steps. One V head of every
    sequence (and a second one of the longest) is recomputed by the oracle as
    one reduced segment (its three channel groups, one K head, one V head)
    over prefill + decode; the fused norm is checked on every output row."""
    wl = gi.workload_varlen()
    shape, w, x = wl["shape"], wl["weights"], wl["inputs"]
    lengths, cu = wl["lengths"], wl["cu_seqlens"]
    T, N, Hk, Hv, D = int(sum(lengths)), len(lengths), 16, 64, 128
    C = shape.qkv_features
    d = gdn.dims(Hk, Hv, D, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    xs, csd, Sd, cud = cuda(x.mixed_qkv), cuda(wl["conv_state"]), cuda(wl["state"]), cuda(cu)
    y = torch.empty_like(xs)
    gdn.gdn_conv_update(d, cud, xs, cuda(w.conv_w), csd, y)
    qk = Hk * D
    core = torch.empty((T, Hv, D), device="cuda")
    out = torch.empty((T, Hv, D), device="cuda", dtype=torch.bfloat16)
    gdn.gdn_prefill_chunked(d, cud, y[:, :qk], y[:, qk:2 * qk], y[:, 2 * qk:], cuda(x.a),
                            cuda(x.b), cuda(w.decay_param), cuda(w.dt_bias), Sd, core_out=core,
                            z=cuda(x.z).view(T, Hv, D), norm_w=cuda(w.norm_w), out=out)
    run = DecodeRunner(shape, w, wl["conv_state"], wl["state"])
    run.conv_state, run.state = csd, Sd
    dec_core = []
    for s in range(16):
        c, _ = run.step(wl["decode"][s], norm=False)
        dec_core.append(c)
    torch.cuda.synchronize()
    core_h = core.cpu()
    dec_h = torch.stack([c.cpu() for c in dec_core])  # [16][N][Hv][D]
    # one V head per sequence (heads spread over the 64, the longest sequence
    # also with a second head), each recomputed by the oracle in parallel
    pairs = [(n, (17 * n + 5) % Hv) for n in range(N)] + [(int(np.argmax(lengths)), 63)]
    X = F64(x.mixed_qkv)
    A, Bb, Z = F64(x.a), F64(x.b), F64(x.z).reshape(T, Hv, D)

    def recompute(pair):
        n, h = pair
        s0, s1 = int(cu[n]), int(cu[n + 1])
        ch = _head_channels(shape, h)
        xs_n = np.concatenate([X[s0:s1][:, ch]] + [F64(wl["decode"][s].mixed_qkv)[n:n + 1][:, ch]
                                                   for s in range(16)])
        a_n = np.concatenate([A[s0:s1, h:h + 1]] + [F64(wl["decode"][s].a)[n:n + 1, h:h + 1]
                                                    for s in range(16)])
        b_n = np.concatenate([Bb[s0:s1, h:h + 1]] + [F64(wl["decode"][s].b)[n:n + 1, h:h + 1]
                                                     for s in range(16)])
        return oracle.segment(
            1, 1, D, 0, shape.decay, xs_n, a_n, b_n, None, F64(w.conv_w)[ch],
            F64(w.decay_param)[h:h + 1], F64(w.dt_bias)[h:h + 1], F64(w.norm_w),
            F64(wl["conv_state"])[n][ch], F64(wl["state"])[n][h:h + 1])

    refs = parallel_map(recompute, pairs)
    Sd_h, csd_h = Sd.cpu(), F64(csd.cpu())
    for (n, h), (rc, _, rcs, rS) in zip(pairs, refs):
        s0, s1 = int(cu[n]), int(cu[n + 1])
        ch = _head_channels(shape, h)
        L = s1 - s0
        tag = f"seq {n} (len {L}) head {h}"
        assert_abs(core_h[s0:s1, h], rc[:L, 0], CHUNK_OUT_ABS, tag + " prefill output")
        assert_abs(dec_h[:, n, h], rc[L:, 0], CHUNK_OUT_ABS, tag + " decode output")
        assert_abs(Sd_h[n, h:h + 1], rS, CHUNK_STATE_ABS, tag + " final state")
        assert np.array_equal(csd_h[n][ch], rcs), tag + " conv state"
    # the fused norm of the whole prefill against the oracle's norm of the
    # kernel's core output
    ry = oracle.gated_rmsnorm(F64(core_h), Z, F64(w.norm_w), 1e-6)
    assert_lowp(out.cpu(), ry, "bf16", "varlen fused norm")
    assert gdn.gdn_device_error() == 0
