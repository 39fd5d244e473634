"""Shared helpers for the GPU parity tests: device upload, oracle references
and the tolerance checks."""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from typing import Callable, Iterable, List, Optional

import numpy as np
import torch

import gdn_inputs as gi
import oracle

F64 = gi.as_f64

# the decode-path bounds (fp32 state): max |d o| and normwise state error
DECODE_OUT_ABS = 1e-4
DECODE_STATE_REL = 1e-5
# the chunked-path bounds with f16/bf16 I/O
CHUNK_OUT_ABS = 0.012
CHUNK_STATE_ABS = 1e-3


def cuda(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().to("cuda")


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the storage dtype at |x| (normal range; floor at the
    smallest subnormal spacing)."""
    ax = np.abs(np.asarray(x, np.float64))
    mant = {"f16": 10, "bf16": 7, "f32": 23}[dtype]
    emin = {"f16": -14, "bf16": -126, "f32": -126}[dtype]
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** emin)))
    return 2.0 ** (np.maximum(e, emin) - mant)


def assert_abs(gpu, ref, tol, what):
    g, r = F64(gpu) if isinstance(gpu, torch.Tensor) else gpu, ref
    assert g.shape == r.shape, (what, g.shape, r.shape)
    err = np.abs(g - r)
    m = float(err.max(initial=0.0))
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    assert m <= tol, f"{what}: max abs err {m:.3e} > {tol:.1e} at {np.unravel_index(err.argmax(), err.shape)}"
    return m


def assert_state_rel(gpu, ref, tol, what, axis_batch=True):
    """max|S_gpu - S_ref| / max|S_ref| per leading index (sequence)."""
    g = F64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    worst = 0.0
    for b in range(g.shape[0]):
        den = max(float(np.abs(ref[b]).max()), 1e-30)
        e = float(np.abs(g[b] - ref[b]).max()) / den
        worst = max(worst, e)
        assert e <= tol, f"{what}[{b}]: normwise state error {e:.3e} > {tol:.1e}"
    return worst


def assert_lowp(gpu, ref, dtype, what, rel=1e-4, abs_floor=None):
    """Low-precision output: |d| <= 1 ulp(dtype, max(|ref|, |gpu|)) + rel*|ref|
    + abs_floor. For fp32 outputs (where one ulp is far below the fp32
    arithmetic error of a near-zero result) abs_floor defaults to 1e-6."""
    if abs_floor is None:
        abs_floor = 1e-6 if dtype == "f32" else 0.0
    g = F64(gpu) if isinstance(gpu, torch.Tensor) else gpu
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    bound = ulp(np.maximum(np.abs(ref), np.abs(g)), dtype) + rel * np.abs(ref) + abs_floor
    err = np.abs(g - ref)
    bad = err > bound
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements beyond 1 ulp; worst "
                           f"{float((err - bound).max()):.3e} at {np.unravel_index((err - bound).argmax(), err.shape)}")


def assert_gated(out_gpu, ref_y, ref_core, z, norm_w, dtype, what, core_gpu=None,
                 eps_o=DECODE_OUT_ABS, rms_eps=1e-6):
    """The gated-RMSNorm output of a fused call, checked two ways:
    (1) if the call also returned its fp32 core output, the epilogue alone:
        against the oracle's gated norm of that very core output, within
        1 ulp + 1e-4 relative;
    (2) against the oracle end to end, with the core output's own error
        bound eps_o carried through the norm: y_j = o_j r w_j silu(z_j) with
        r = (mean o^2 + eps)^(-1/2) moves by at most about
        eps_o r |w_j silu(z_j)| through o_j and as much again through r."""
    zf, wf = F64(z) if isinstance(z, torch.Tensor) else z, F64(norm_w) if isinstance(
        norm_w, torch.Tensor) else norm_w
    zf = zf.reshape(ref_y.shape)
    if core_gpu is not None:
        cg = F64(core_gpu) if isinstance(core_gpu, torch.Tensor) else core_gpu
        assert_lowp(out_gpu, oracle.gated_rmsnorm(cg, zf, wf, rms_eps), dtype, what + " (epilogue)")
    r = 1.0 / np.sqrt(np.mean(ref_core * ref_core, axis=-1, keepdims=True) + rms_eps)
    gate = np.abs(wf * (zf / (1.0 + np.exp(-zf))))
    g = F64(out_gpu) if isinstance(out_gpu, torch.Tensor) else out_gpu
    bound = (ulp(np.maximum(np.abs(ref_y), np.abs(g)), dtype) + 1e-4 * np.abs(ref_y)
             + 2.0 * eps_o * r * gate + (1e-6 if dtype == "f32" else 0.0))
    err = np.abs(g - ref_y)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    bad = err > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond the carried bound"


def dtype_name(t: torch.dtype) -> str:
    return {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}[t]


def decode_reference(shape: gi.Shape, w: gi.Weights, x: gi.StepInputs, conv_state: np.ndarray,
                     S: np.ndarray, seqs=None, with_norm=True):
    """Oracle O6 for one decode token of each sequence in ``seqs`` (all if
    None): returns core [n][Hv][D], y (or None), new conv states, new states."""
    B = x.mixed_qkv.shape[0]
    seqs = list(range(B)) if seqs is None else list(seqs)
    X, A, Bb, Z = F64(x.mixed_qkv), F64(x.a), F64(x.b), F64(x.z)
    cw, dp, dt, nw = F64(w.conv_w), F64(w.decay_param), F64(w.dt_bias), F64(w.norm_w)
    cores, ys, css, Ss = [], [], [], []
    for i, b in enumerate(seqs):
        core, y, cs, St = oracle.segment(
            shape.n_k_heads, shape.n_v_heads, shape.head_dim, shape.map, shape.decay,
            X[b:b + 1], A[b:b + 1], Bb[b:b + 1], Z[b:b + 1] if with_norm else None, cw, dp, dt,
            nw, conv_state[i], S[i])
        cores.append(core[0])
        ys.append(y[0] if y is not None else None)
        css.append(cs)
        Ss.append(St)
    return (np.stack(cores), np.stack(ys) if with_norm else None, np.stack(css), np.stack(Ss))


class DecodeRunner:
    """Holds device tensors for repeated decode steps through the binding."""

    def __init__(self, shape: gi.Shape, w: gi.Weights, conv_state: torch.Tensor,
                 state: torch.Tensor):
        import gated_delta_net_causal_gb300 as gdn
        self.gdn = gdn
        self.shape = shape
        self.d = gdn.dims(shape.n_k_heads, shape.n_v_heads, shape.head_dim, shape.map,
                          shape.decay, gi.DTYPES[shape.dtype])
        self.w = {k: cuda(getattr(w, k)) for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
        self.conv_state = cuda(conv_state)
        self.state = cuda(state)

    def step(self, x: gi.StepInputs, core=True, norm=True):
        B, Hv, D = x.mixed_qkv.shape[0], self.shape.n_v_heads, self.shape.head_dim
        io = gi.DTYPES[self.shape.dtype]
        core_out = torch.full((B, Hv, D), float("nan"), device="cuda") if core else None
        out = torch.full((B, Hv, D), float("nan"), device="cuda", dtype=io) if norm else None
        z = cuda(x.z).view(B, Hv, D) if norm else None
        self.gdn.gdn_decode_step(self.d, cuda(x.mixed_qkv), cuda(x.a), cuda(x.b),
                                 self.w["decay_param"], self.w["dt_bias"], self.w["conv_w"],
                                 self.conv_state, self.state, core_out=core_out, z=z,
                                 norm_w=self.w["norm_w"] if norm else None, out=out)
        return core_out, out


def parallel_map(fn: Callable, items: Iterable) -> List:
    """fn over items on the host's cores: the oracle runs in C through ctypes,
    which releases the interpreter lock, so threads run it in parallel."""
    items = list(items)
    with ThreadPoolExecutor(max_workers=min(len(items), os.cpu_count() or 4) or 1) as ex:
        return list(ex.map(fn, items))
