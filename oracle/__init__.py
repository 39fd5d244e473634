"""fp64 CPU oracle for the gated delta-net core -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's
``cpu_baseline`` / ``--impl reference`` legs may import this package. The
library's product path never imports it, and it imports nothing from the
library: the two share no code. The arithmetic lives in ``gdn_oracle.c``
(plain scalar double-precision loops, one function per step of the method,
each citing the page it restates); this module compiles it with gcc and
marshals numpy float64 arrays to it through ctypes.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against values the pages print (the scalar worked example, the head-map
example, the l2-normalise example), closed forms, library routines
(numpy.convolve, numpy.linalg) and the five recurrence properties. The pages'
fingerprinted tolerance contracts (the Metal test's numerical_tolerance ids)
print no values, so nothing can be pinned to them.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

GROUPED, TILED = 0, 1
LOG_RATE, NEGATIVE_RATE = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction, so x86
    and Arm hosts give identical results)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_INT = ctypes.c_int
_DBL = ctypes.c_double


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            L.gdn_oracle_sigmoid.restype = _DBL
            L.gdn_oracle_sigmoid.argtypes = [_DBL]
            L.gdn_oracle_silu.restype = _DBL
            L.gdn_oracle_silu.argtypes = [_DBL]
            L.gdn_oracle_softplus.restype = _DBL
            L.gdn_oracle_softplus.argtypes = [_DBL]
            L.gdn_oracle_k_head.restype = _INT
            L.gdn_oracle_k_head.argtypes = [_INT, _INT, _INT, _INT]
            L.gdn_oracle_conv.restype = None
            L.gdn_oracle_conv.argtypes = [_I64, _I32, _D, _D, _D, _D]
            L.gdn_oracle_l2norm_rows.restype = None
            L.gdn_oracle_l2norm_rows.argtypes = [_I64, _I32, _DBL, _D]
            L.gdn_oracle_l2norm_rows_clamped.restype = None
            L.gdn_oracle_l2norm_rows_clamped.argtypes = [_I64, _I32, _DBL, _D]
            L.gdn_oracle_gates.restype = None
            L.gdn_oracle_gates.argtypes = [_I64, _I32, _INT, _D, _D, _D, _D, _D, _D]
            L.gdn_oracle_delta.restype = None
            L.gdn_oracle_delta.argtypes = [_I32, _I32, _I32, _INT, _I64, _D, _D, _D, _D, _D, _D, _D]
            L.gdn_oracle_gated_rmsnorm.restype = None
            L.gdn_oracle_gated_rmsnorm.argtypes = [_I64, _I32, _DBL, _D, _D, _D, _D]
            L.gdn_oracle_segment.restype = None
            L.gdn_oracle_segment.argtypes = [_I32, _I32, _I32, _INT, _INT, _DBL, _INT, _DBL, _I64,
                                             _D, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D, _D]
            L.gdn_oracle_delta_chunked.restype = None
            L.gdn_oracle_delta_chunked.argtypes = [_I32, _I32, _I32, _INT, _I64, _I32, _D, _D, _D,
                                                   _D, _D, _D, _D]
            L.gdn_oracle_delta_affine.restype = None
            L.gdn_oracle_delta_affine.argtypes = [_I32, _I32, _I32, _INT, _I64, _I32, _D, _D, _D,
                                                  _D, _D, _D, _D]
            L.gdn_oracle_chunk_factors.restype = None
            L.gdn_oracle_chunk_factors.argtypes = [_I32, _I32, _I32, _INT, _I64, _I32, _I32, _D,
                                                   _D, _D, _D, _D, _D, _D, _D, _D]
            L.gdn_oracle_delta_bruteforce.restype = _INT
            L.gdn_oracle_delta_bruteforce.argtypes = [_I32, _I32, _I32, _INT, _I64, _D, _D, _D,
                                                      _D, _D, _D, _D]
            _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: Optional[np.ndarray]):
    if a is None:
        return ctypes.cast(None, _D)
    assert a.dtype == np.float64 and a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(_D)


# ----------------------------------------------------------------- scalars

def sigmoid(x: float) -> float:
    return lib().gdn_oracle_sigmoid(float(x))


def silu(x: float) -> float:
    return lib().gdn_oracle_silu(float(x))


def softplus(x: float) -> float:
    return lib().gdn_oracle_softplus(float(x))


def k_head(map_: int, h: int, n_k: int, n_v: int) -> int:
    return lib().gdn_oracle_k_head(map_, h, n_k, n_v)


# -------------------------------------------------------------------- steps

def conv(x, w, state) -> Tuple[np.ndarray, np.ndarray]:
    """O1 over one sequence: x [T][C], w [C][4], state [C][3] -> (y, new state)."""
    x, w, st = _f64(x), _f64(w), _f64(state).copy()
    T, C = x.shape
    y = np.zeros((T, C))
    lib().gdn_oracle_conv(T, C, _p(x), _p(w), _p(st), _p(y))
    return y, st


def conv_varlen(x, w, states, cu_seqlens) -> Tuple[np.ndarray, np.ndarray]:
    """O1 per sequence of a packed batch: x [T_tot][C], states [N][C][3]."""
    x = _f64(x)
    cu = [int(c) for c in np.asarray(cu_seqlens)]
    ys, sts = [], []
    for n in range(len(cu) - 1):
        y, st = conv(x[cu[n]:cu[n + 1]], w, np.asarray(states)[n])
        ys.append(y)
        sts.append(st)
    return np.concatenate(ys, 0) if ys else np.zeros((0, x.shape[1])), np.stack(sts)


def l2norm(x, eps: float = 1e-6, clamped: bool = False) -> np.ndarray:
    """O2 along the last axis."""
    y = _f64(x).copy()
    width = y.shape[-1]
    rows = y.size // width if width else 0
    fn = lib().gdn_oracle_l2norm_rows_clamped if clamped else lib().gdn_oracle_l2norm_rows
    fn(rows, width, float(eps), _p(y))
    return y


def gates(a, b, decay_param, dt_bias, decay: int) -> Tuple[np.ndarray, np.ndarray]:
    """O3: a, b [T][Hv] -> (g, beta)."""
    a, b = _f64(a), _f64(b)
    T, Hv = a.shape
    g, beta = np.zeros((T, Hv)), np.zeros((T, Hv))
    lib().gdn_oracle_gates(T, Hv, decay, _p(_f64(decay_param)), _p(_f64(dt_bias)), _p(a), _p(b),
                           _p(g), _p(beta))
    return g, beta


def _delta_common(fn, q, k, v, g, beta, S, map_: int, *extra):
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    S = _f64(S).copy()
    T, Hk, D = q.shape
    Hv = v.shape[1]
    o = np.zeros((T, Hv, D))
    r = fn(Hk, Hv, D, map_, T, *extra, _p(q), _p(k), _p(v), _p(g), _p(beta), _p(S), _p(o))
    if r not in (None, 0):
        raise ValueError("oracle rejected the shape")
    return o, S


def delta(q, k, v, g, beta, S, map_: int):
    """O4, the token recurrence: q, k [T][Hk][D] normalised; v [T][Hv][D];
    g, beta [T][Hv]; S [Hv][D][D]. Returns (o, S_new)."""
    return _delta_common(lib().gdn_oracle_delta, q, k, v, g, beta, S, map_)


def delta_chunked(q, k, v, g, beta, S, map_: int, chunk: int = 64):
    """O7, the chunk-wise summation of O4."""
    return _delta_common(lib().gdn_oracle_delta_chunked, q, k, v, g, beta, S, map_, int(chunk))


def delta_affine(q, k, v, g, beta, S, map_: int, chunk: int = 64):
    """O9, O4 carried chunk by chunk as affine maps of the chunk-start state:
    o = X S^T + Y, then S <- S M + N (factors from chunk_factors)."""
    return _delta_common(lib().gdn_oracle_delta_affine, q, k, v, g, beta, S, map_, int(chunk))


def chunk_factors(q, k, v, g, beta, map_: int, h: int, t0: int, L: int):
    """O9's per-chunk factors for V head h over tokens [t0, t0 + L): returns
    (M [D][D], N [D][D], X [L][D], Y [L][D]) with S_end = S0 M + N and the
    chunk's outputs X S0^T + Y (S0 = the state before token t0)."""
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    T, Hk, D = q.shape
    Hv = v.shape[1]
    if not (0 <= t0 and 1 <= L and t0 + L <= T and 0 <= h < Hv):
        raise ValueError("chunk outside the sequence")
    M, N = np.zeros((D, D)), np.zeros((D, D))
    X, Y = np.zeros((L, D)), np.zeros((L, D))
    lib().gdn_oracle_chunk_factors(Hk, Hv, D, map_, int(t0), int(L), int(h), _p(q), _p(k),
                                   _p(v), _p(g), _p(beta), _p(M), _p(N), _p(X), _p(Y))
    return M, N, X, Y


def delta_bruteforce(q, k, v, g, beta, S, map_: int):
    """O8, explicit matrix products in long double (D <= 8)."""
    return _delta_common(lib().gdn_oracle_delta_bruteforce, q, k, v, g, beta, S, map_)


def gated_rmsnorm(o, z, w, eps: float = 1e-6) -> np.ndarray:
    """O5 along the last axis of o [..][D]."""
    o, z, w = _f64(o), _f64(z), _f64(w)
    D = o.shape[-1]
    y = np.zeros_like(o)
    lib().gdn_oracle_gated_rmsnorm(o.size // D, D, float(eps), _p(o), _p(z), _p(w), _p(y))
    return y


def segment(Hk: int, Hv: int, D: int, map_: int, decay: int, mixed_qkv, a, b, z, conv_w,
            decay_param, dt_bias, norm_w, conv_state, S, l2_eps: float = 1e-6,
            rms_eps: float = 1e-6, l2_clamped: bool = False):
    """O6 over one sequence: returns (core [T][Hv][D], y or None, conv_state, S)."""
    x = _f64(mixed_qkv)
    T = x.shape[0]
    a, b = _f64(a).reshape(T, Hv), _f64(b).reshape(T, Hv)
    zz = None if z is None else _f64(z).reshape(T, Hv, D)
    cs = _f64(conv_state).copy()
    St = _f64(S).copy()
    core = np.zeros((T, Hv, D))
    y = None if z is None else np.zeros((T, Hv, D))
    lib().gdn_oracle_segment(Hk, Hv, D, map_, decay, float(l2_eps), 1 if l2_clamped else 0,
                             float(rms_eps), T, _p(x), _p(a), _p(b), _p(zz), _p(_f64(conv_w)),
                             _p(_f64(decay_param)), _p(_f64(dt_bias)), _p(_f64(norm_w)), _p(cs),
                             _p(St), _p(core), _p(y))
    return core, y, cs, St


def prefill_core(Hk: int, Hv: int, D: int, map_: int, q, k, v, g, beta, S, cu_seqlens,
                 l2_eps: Optional[float] = 1e-6):
    """O2 + O4 over a packed batch whose q/k/v are already convolved, with
    gates already formed. Each sequence n runs from its own S[n]. l2_eps=None
    means q/k are used as given (already normalised)."""
    cu = [int(c) for c in np.asarray(cu_seqlens)]
    q = _f64(q)
    k = _f64(k)
    if l2_eps is not None:
        q = l2norm(q, l2_eps)
        k = l2norm(k, l2_eps)
    v, g, beta = _f64(v), _f64(g), _f64(beta)
    S = _f64(S).copy()
    o = np.zeros(v.shape)
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        o[s:e], S[n] = delta(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], S[n], map_)
    return o, S


def round_bf16(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), via float32: the cast
    the page's Linear applies to its output (`astype` to the input dtype)."""
    f = np.ascontiguousarray(_f64(x), dtype=np.float64).astype(np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64).reshape(np.shape(x))


def linear(x, w, bias=None, round_out: bool = True) -> np.ndarray:
    """y = x w^T (+ bias), the page's `Linear::forward` (libmir-metal
    decode/mod.rs): a matmul in fp64 (a library routine), the bias, then one
    rounding to bf16 (reading: the bias joins before the single cast)."""
    y = _f64(x) @ _f64(w).T
    if bias is not None:
        y = y + _f64(bias)
    return round_bf16(y) if round_out else y


def decode_layer(Hk: int, Hv: int, D: int, map_: int, decay: int, x, w_in, b_in, w_out, b_out, conv_w,
                 decay_param, dt_bias, norm_w, conv_state, S, l2_eps: float = 1e-6,
                 rms_eps: float = 1e-6):
    """One decode step of a layer, in the page's order (libmir-metal
    decode/mod.rs, `build`): the qkv, gate, beta and alpha projections of
    the input x [B][hidden] (rows of w_in: qkv | z | b | a), each rounded to
    bf16; per sequence the core (O6 with its gated RMSNorm), its output
    rounded to bf16; the output projection, rounded to bf16. Returns
    (y [B][hidden], conv_state, S, y_core [B][Hv][D])."""
    x = _f64(x)
    B = x.shape[0]
    C = (2 * Hk + Hv) * D
    vw = Hv * D
    proj = linear(x, w_in[:C + vw + 2 * Hv], None if b_in is None else _f64(b_in)[:C + vw + 2 * Hv])
    qkv, z = proj[:, :C], proj[:, C:C + vw]
    bb, aa = proj[:, C + vw:C + vw + Hv], proj[:, C + vw + Hv:C + vw + 2 * Hv]
    cs, St = _f64(conv_state).copy(), _f64(S).copy()
    yc = np.zeros((B, Hv, D))
    for n in range(B):
        _, y, cs[n], St[n] = segment(Hk, Hv, D, map_, decay, qkv[n:n + 1], aa[n:n + 1], bb[n:n + 1],
                                     z[n:n + 1], conv_w, decay_param, dt_bias, norm_w, cs[n], St[n],
                                     l2_eps=l2_eps, rms_eps=rms_eps)
        yc[n] = round_bf16(y[0])
    out = linear(yc.reshape(B, vw), w_out, b_out)
    return out, cs, St, yc


__all__ = ["build", "lib", "sigmoid", "silu", "softplus", "k_head", "conv", "conv_varlen",
           "l2norm", "gates", "delta", "delta_chunked", "delta_affine", "chunk_factors",
           "delta_bruteforce", "gated_rmsnorm",
           "segment", "prefill_core", "round_bf16", "linear", "decode_layer", "GROUPED", "TILED", "LOG_RATE", "NEGATIVE_RATE"]
