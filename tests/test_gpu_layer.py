"""The decode layer (NEXT-2): gdn_linear (the tcgen05 projections) against
the oracle's fp64 matmul, and gdn_decode_layer -- the fused input projection,
the core with its gated RMSNorm, the output projection (libmir-metal
decode/mod.rs, `build`) -- checked three ways: bit for bit against the same
three calls made one by one, each stage against the oracle on the GPU's own
inputs to it, and end to end against oracle.decode_layer."""

import numpy as np
import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
import gdn_inputs as gi
import oracle
from tests.gpu_helpers import DECODE_OUT_ABS, DECODE_STATE_REL, F64, assert_gated, cuda, ulp

BF = torch.bfloat16


def _bf(g, shape, std):
    return gi.to_dtype(gi.normal(g, shape, std), "bf16")


def _assert_linear(y_gpu, x, w, bias, what):
    """|y - ref| <= 1 ulp(bf16) + the fp32 accumulation bound K 2^-23 |x||w|^T."""
    ref = oracle.linear(F64(x), F64(w), None if bias is None else F64(bias))
    K = x.shape[1]
    acc_bound = K * 2.0 ** -23 * (np.abs(F64(x)) @ np.abs(F64(w)).T)
    g = F64(y_gpu)
    bound = ulp(np.maximum(np.abs(ref), np.abs(g)), "bf16") + acc_bound
    err = np.abs(g - ref)
    assert np.all(np.isfinite(g)), what
    assert (err <= bound).all(), f"{what}: {int((err > bound).sum())} elements out of bound"


@pytest.mark.gpu
@pytest.mark.parametrize("M,N,K,with_bias,pad", [(1, 128, 64, False, 0), (3, 192, 256, True, 8),
                                                  (64, 12352, 2048, False, 0), (64, 2048, 4096, True, 0),
                                                  (128, 256, 512, False, 24), (17, 64, 1024, True, 0),
                                                  (31, 2048, 4096, True, 0), (32, 2048, 4096, False, 8),
                                                  (33, 12352, 2048, True, 0)])
def test_linear_matches_the_oracle(M, N, K, with_bias, pad):
    """Shapes of the fused input projection (N=12352), the split-K output
    projection (N=2048, K=4096), the MMA's full 128 rows, a single row,
    strided rows of x and y, and row counts on both sides of the switch
    between the two ring sizes (32 rows)."""
    g = gi.rng(100 + M + N + K)
    x = _bf(g, (M, K + pad), 1.0)
    w = _bf(g, (N, K), 1.0 / np.sqrt(K))
    bias = torch.from_numpy(gi.normal(g, (N,), 1.0).astype(np.float32)) if with_bias else None
    y = torch.full((M, N + pad), float("nan"), device="cuda", dtype=BF)
    gdn.gdn_linear(cuda(x)[:, :K], cuda(w), y[:, :N], bias=None if bias is None else cuda(bias))
    torch.cuda.synchronize()
    _assert_linear(y[:, :N].cpu(), x[:, :K], w, bias, f"linear {M}x{N}x{K}")
    if pad:
        assert torch.isnan(y[:, N:].float()).all()  # the padding columns are untouched
    assert gdn.gdn_device_error() == 0


def _layer_case(seed, Hk, Hv, D, hidden, B, biases):
    g = gi.rng(seed)
    shape = gi.Shape(Hk, Hv, D, map=gi.GROUPED, decay=gi.LOG_RATE, dtype="bf16")
    C, vw = (2 * Hk + Hv) * D, Hv * D
    n_in = (C + vw + 2 * Hv + 63) // 64 * 64
    w = gi.layer_weights(g, shape)
    t = dict(
        x=_bf(g, (B, hidden), 1.0),
        w_in=_bf(g, (n_in, hidden), 1.0 / np.sqrt(hidden)),
        w_out=_bf(g, (hidden, vw), 1.0 / np.sqrt(vw)),
        b_in=torch.from_numpy(gi.normal(g, (n_in,), 0.1).astype(np.float32)) if biases else None,
        b_out=torch.from_numpy(gi.normal(g, (hidden,), 0.1).astype(np.float32)) if biases else None,
        conv_state=gi.to_dtype(gi.normal(g, (B, C, 3), 0.1), "bf16"),
        state=gi.delta_state(g, shape, B, std=0.02))
    return shape, w, t, C, vw, n_in


def _run_layer(d, hidden, w, t):
    cs, st = cuda(t["conv_state"]), cuda(t["state"])
    y = torch.full((t["x"].shape[0], hidden), float("nan"), device="cuda", dtype=BF)
    opt = lambda v: None if v is None else cuda(v)
    gdn.gdn_decode_layer(d, cuda(t["x"]), cuda(t["w_in"]), cuda(t["w_out"]), cuda(w.conv_w),
                         cuda(w.decay_param), cuda(w.dt_bias), cuda(w.norm_w), cs, st, y,
                         b_in=opt(t["b_in"]), b_out=opt(t["b_out"]))
    torch.cuda.synchronize()
    return y, cs, st


@pytest.mark.gpu
@pytest.mark.parametrize("Hk,Hv,D,hidden,B,biases", [(2, 8, 64, 128, 3, True),
                                                     (16, 32, 128, 2048, 64, False),
                                                     (16, 32, 128, 2048, 1, True),
                                                     (4, 16, 96, 512, 32, True)])
def test_decode_layer(Hk, Hv, D, hidden, B, biases):
    shape, w, t, C, vw, n_in = _layer_case(700 + B + Hk, Hk, Hv, D, hidden, B, biases)
    d = gdn.dims(Hk, Hv, D, map=shape.map, decay=shape.decay, io_dtype=BF)
    y, cs, st = _run_layer(d, hidden, w, t)
    assert gdn.gdn_device_error() == 0

    # (1) bit for bit the three calls made one by one
    opt = lambda v: None if v is None else cuda(v)
    proj = torch.empty((B, n_in), device="cuda", dtype=BF)
    gdn.gdn_linear(cuda(t["x"]), cuda(t["w_in"]), proj, bias=opt(t["b_in"]))
    qkv = proj[:, :C].contiguous()
    z = proj[:, C:C + vw].contiguous()
    bb = proj[:, C + vw:C + vw + Hv].contiguous()
    aa = proj[:, C + vw + Hv:C + vw + 2 * Hv].contiguous()
    cs2, st2 = cuda(t["conv_state"]), cuda(t["state"])
    core = torch.empty((B, Hv, D), device="cuda")
    yc = torch.empty((B, Hv, D), device="cuda", dtype=BF)
    gdn.gdn_decode_step(d, qkv, aa, bb, cuda(w.decay_param), cuda(w.dt_bias), cuda(w.conv_w), cs2, st2,
                        core_out=core, z=z, norm_w=cuda(w.norm_w), out=yc)
    y2 = torch.empty((B, hidden), device="cuda", dtype=BF)
    gdn.gdn_linear(yc.view(B, vw), cuda(t["w_out"]), y2, bias=opt(t["b_out"]))
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), y2.cpu())
    assert torch.equal(cs.cpu(), cs2.cpu()) and torch.equal(st.cpu(), st2.cpu())

    # (2) each stage against the oracle on the GPU's own inputs to it
    _assert_linear(proj.cpu(), t["x"], t["w_in"], t["b_in"], "input projection")
    rc, ry, rcs, rS = [], [], [], []
    for n in range(B):
        c_n, y_n, cs_n, S_n = oracle.segment(Hk, Hv, D, shape.map, shape.decay, F64(qkv[n:n + 1].cpu()),
                                             F64(aa[n:n + 1].cpu()), F64(bb[n:n + 1].cpu()),
                                             F64(z[n:n + 1].cpu()), F64(w.conv_w), F64(w.decay_param),
                                             F64(w.dt_bias), F64(w.norm_w), F64(t["conv_state"][n]),
                                             F64(t["state"][n]))
        rc.append(c_n[0]), ry.append(y_n[0]), rcs.append(cs_n), rS.append(S_n)
    assert_gated(yc.cpu(), np.stack(ry), np.stack(rc), z.cpu().view(B, Hv, D), w.norm_w, "bf16",
                 "layer core gated output", core_gpu=core.cpu(), eps_o=DECODE_OUT_ABS)
    assert np.array_equal(F64(cs.cpu()), np.stack(rcs))  # the conv state holds raw projected inputs
    rS = np.stack(rS)
    assert np.linalg.norm(F64(st.cpu()) - rS) <= DECODE_STATE_REL * np.linalg.norm(rS)
    _assert_linear(y.cpu(), yc.cpu().view(B, vw), t["w_out"], t["b_out"], "output projection")

    # (3) end to end against oracle.decode_layer: the GPU's projections differ
    # from the oracle's by at most one bf16 rounding (and fp32 sums), which the
    # core carries on; bounded loosely as a relative error
    oy, _, _, _ = oracle.decode_layer(Hk, Hv, D, shape.map, shape.decay, F64(t["x"]), F64(t["w_in"]),
                                      None if t["b_in"] is None else F64(t["b_in"]), F64(t["w_out"]),
                                      None if t["b_out"] is None else F64(t["b_out"]), F64(w.conv_w),
                                      F64(w.decay_param), F64(w.dt_bias), F64(w.norm_w), F64(t["conv_state"]),
                                      F64(t["state"]))
    rel = np.linalg.norm(F64(y.cpu()) - oy) / np.linalg.norm(oy)
    assert rel < 2e-2, rel
