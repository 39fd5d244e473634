"""Seeded synthetic inputs for the gated delta-net core.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests. It holds no arithmetic of the method itself: it only draws
random numbers (numpy PCG64, fixed seeds), rounds them once to the storage
dtype (round-to-nearest-even, done by torch's dtype cast) and lays them out
in the shapes the library calls take.

Every array is returned twice over: as a CPU torch tensor in its storage
dtype (what the GPU side uploads) and implicitly as the exact float64 value
of that tensor (``as_f64``), which is what the oracle consumes. The cast
from bf16/f16/f32 to float64 is exact, so both sides see identical numbers.

Distribution notation: ``N(0, s)`` takes ``s`` as the standard deviation,
``U(a, b)`` is uniform on [a, b).
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np
import torch

GROUPED = 0
TILED = 1
LOG_RATE = 0
NEGATIVE_RATE = 1

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _round_to_odd_f32(x: torch.Tensor) -> torch.Tensor:
    """float64 -> float32 rounded to odd: truncate toward zero, then set the
    last mantissa bit when anything was dropped. A second rounding (to
    nearest even) of the result to a format at least two bits narrower gives
    exactly the once-rounded float64 value (the round-to-odd theorem), so the
    16-bit conversions below round once although they pass through float32."""
    f = x.to(torch.float32)
    away = f.to(torch.float64).abs() > x.abs()
    f = torch.where(away, torch.nextafter(f, torch.zeros_like(f)), f)
    inexact = (f.to(torch.float64) != x).to(torch.int32)
    return (f.view(torch.int32) | inexact).view(torch.float32)


def to_dtype(x: np.ndarray, dtype: str) -> torch.Tensor:
    """Round float64 values once, to nearest with ties to even, to the storage
    dtype (finite values in the float32 range)."""
    x = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    if dtype == "f32":
        return x.to(torch.float32)
    return _round_to_odd_f32(x).to(DTYPES[dtype])


def as_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a CPU tensor (any float dtype)."""
    return np.ascontiguousarray(t.detach().to("cpu", torch.float64).numpy())


def normal(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return g.standard_normal(size=shape) * std


def uniform(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape)


def sin_values(n: int, frequency: float, amplitude: float) -> np.ndarray:
    """``sin(i * frequency) * amplitude`` for i in [0, n), evaluated in float32
    like the deterministic fill of the ferrum-kernels gated-delta test
    (``half_values`` / ``float_values``)."""
    i = np.arange(n, dtype=np.float32)
    return (np.sin(i * np.float32(frequency)) * np.float32(amplitude)).astype(np.float64)


@dataclasses.dataclass
class Shape:
    n_k_heads: int
    n_v_heads: int
    head_dim: int
    map: int = GROUPED
    decay: int = LOG_RATE
    dtype: str = "bf16"

    @property
    def qk_features(self) -> int:
        return self.n_k_heads * self.head_dim

    @property
    def v_features(self) -> int:
        return self.n_v_heads * self.head_dim

    @property
    def qkv_features(self) -> int:
        return 2 * self.qk_features + self.v_features

    @property
    def state_len(self) -> int:
        return self.n_v_heads * self.head_dim * self.head_dim


@dataclasses.dataclass
class Weights:
    """Per-layer static parameters (storage dtypes as the library takes them)."""

    conv_w: torch.Tensor  # [C_qkv][4], io dtype
    decay_param: torch.Tensor  # [Hv] f32: A_log (log-rate) or the negative rate
    dt_bias: torch.Tensor  # [Hv] f32
    norm_w: torch.Tensor  # [D] f32


def layer_weights(g: np.random.Generator, shape: Shape, *, a_log: Optional[np.ndarray] = None,
                  dt_bias: Optional[np.ndarray] = None, conv_std: float = 0.16) -> Weights:
    """Default parameter recipe for the configs whose pages give none:
    A_log = ln U[1,16], dt_bias ~ U(-0.5, 0.5), conv weight ~ N(0, 0.16),
    norm weight w_j = 0.82 + 0.013 j. The negative-rate form draws its rate
    as -U[1,16] directly (the same law as -exp(A_log))."""
    C, Hv, D = shape.qkv_features, shape.n_v_heads, shape.head_dim
    conv_w = to_dtype(normal(g, (C, 4), conv_std), shape.dtype)
    u = uniform(g, (Hv,), 1.0, 16.0)
    if a_log is None:
        param = np.log(u) if shape.decay == LOG_RATE else -u
    else:
        param = a_log if shape.decay == LOG_RATE else -np.exp(a_log)
    if dt_bias is None:
        dt_bias = uniform(g, (Hv,), -0.5, 0.5)
    norm_w = 0.82 + 0.013 * np.arange(D, dtype=np.float64)
    return Weights(conv_w=conv_w,
                   decay_param=to_dtype(np.asarray(param, np.float64), "f32"),
                   dt_bias=to_dtype(np.asarray(dt_bias, np.float64), "f32"),
                   norm_w=to_dtype(norm_w, "f32"))


@dataclasses.dataclass
class StepInputs:
    """Per-token activations for a batch of tokens (decode: one per sequence)."""

    mixed_qkv: torch.Tensor  # [T][C_qkv] io dtype, pre-conv
    a: torch.Tensor  # [T][Hv] io dtype (raw alpha input)
    b: torch.Tensor  # [T][Hv] io dtype (raw beta input)
    z: torch.Tensor  # [T][Hv*D] io dtype (output gate input)


def step_inputs(g: np.random.Generator, shape: Shape, tokens: int, *, qkv_std=1.0, ab_std=1.0,
                z_std=1.0) -> StepInputs:
    C, Hv, D = shape.qkv_features, shape.n_v_heads, shape.head_dim
    return StepInputs(
        mixed_qkv=to_dtype(normal(g, (tokens, C), qkv_std), shape.dtype),
        a=to_dtype(normal(g, (tokens, Hv), ab_std), shape.dtype),
        b=to_dtype(normal(g, (tokens, Hv), ab_std), shape.dtype),
        z=to_dtype(normal(g, (tokens, Hv * D), z_std), shape.dtype),
    )


def delta_state(g: np.random.Generator, shape: Shape, batch: int, std: float = 0.02,
                uniform_half_width: Optional[float] = None) -> torch.Tensor:
    n = (batch, shape.n_v_heads, shape.head_dim, shape.head_dim)
    if uniform_half_width is not None:
        x = uniform(g, n, -uniform_half_width, uniform_half_width)
    else:
        x = normal(g, n, std)
    return to_dtype(x, "f32")


def conv_state(g: np.random.Generator, shape: Shape, batch: int, std: float = 0.1,
               uniform_half_width: Optional[float] = None) -> torch.Tensor:
    n = (batch, shape.qkv_features, 3)
    if uniform_half_width is not None:
        x = uniform(g, n, -uniform_half_width, uniform_half_width)
    else:
        x = normal(g, n, std)
    return to_dtype(x, shape.dtype)


def cu_seqlens(lengths: List[int]) -> torch.Tensor:
    return torch.tensor(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))


def varlen_lengths(seed: int, n: int, lo: int, hi: int) -> List[int]:
    """Sequence lengths drawn U[lo, hi] (integers, inclusive), used as drawn."""
    return [int(x) for x in rng(seed).integers(lo, hi + 1, size=n)]


# --------------------------------------------------------------------------
# The five synthetic workloads (seed 20261200 + i for workload i).
# --------------------------------------------------------------------------

SEED_BASE = 20261200


def workload_single_layer_b1(dtype: str = "f16", map: int = GROUPED,
                             decay: int = LOG_RATE) -> Dict:
    """Batch 1, 4 tokens, Hk=16, Hv=32, D=128, f16. mixed_qkv ~N(0,0.25),
    a/b ~N(0,1), z ~N(0,1), conv weight ~N(0,0.16), conv state ~U(-0.04,0.04),
    A_log_h = -1.7 + 0.07 h, dt_bias_h = -0.25 + 0.04 h, norm w_j = 0.82 +
    0.013 j, delta state ~U(-0.025, 0.025)."""
    shape = Shape(16, 32, 128, map=map, decay=decay, dtype=dtype)
    g = rng(SEED_BASE + 1)
    a_log = -1.7 + 0.07 * np.arange(32)
    dt_bias = -0.25 + 0.04 * np.arange(32)
    w = layer_weights(g, shape, a_log=a_log, dt_bias=dt_bias, conv_std=0.16)
    x = step_inputs(g, shape, 4, qkv_std=0.25)
    return dict(shape=shape, weights=w, inputs=x,
                conv_state=conv_state(g, shape, 1, uniform_half_width=0.04),
                state=delta_state(g, shape, 1, uniform_half_width=0.025))


def workload_single_layer_sin(map: int = GROUPED, decay: int = LOG_RATE) -> Dict:
    """The batch-1, 4-token layer on the deterministic fill of the Metal
    conformance test (ferrum-kernels gated_delta_attention_tests.rs, the
    conformance setup: ``half_values`` / ``float_values``, sin(i f) a in
    float32): mixed_qkv (f 0.017, a 0.21), a (0.071, 0.18), b (0.053, 0.24),
    z (0.029, 0.31), conv weight (0.011, 0.16) and conv state (0.023, 0.04)
    in f16, the delta state (0.007, 0.025) in f32, laid out as this
    library's arrays; A_log_h = -1.7 + 0.07 h (its negative rate -exp(A_log)
    in float32), dt_bias_h = -0.25 + 0.04 h, norm w_j = 0.82 + 0.013 j."""
    shape = Shape(16, 32, 128, map=map, decay=decay, dtype="f16")
    T, C, Hv, D = 4, shape.qkv_features, shape.n_v_heads, shape.head_dim

    def h16(n, f, a, *dims):
        return to_dtype(sin_values(n, f, a), "f16").view(*dims)
    x = StepInputs(mixed_qkv=h16(T * C, 0.017, 0.21, T, C), a=h16(T * Hv, 0.071, 0.18, T, Hv),
                   b=h16(T * Hv, 0.053, 0.24, T, Hv), z=h16(T * Hv * D, 0.029, 0.31, T, Hv * D))
    idx = np.arange(Hv, dtype=np.float32)
    log_rates = np.float32(-1.7) + idx * np.float32(0.07)
    param = log_rates if decay == LOG_RATE else -np.exp(log_rates)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    w = Weights(conv_w=h16(C * 4, 0.011, 0.16, C, 4), decay_param=f32(param),
                dt_bias=f32(np.float32(-0.25) + idx * np.float32(0.04)),
                norm_w=f32(np.float32(0.82) + np.arange(D, dtype=np.float32) * np.float32(0.013)))
    state = f32(sin_values(Hv * D * D, 0.007, 0.025)).view(1, Hv, D, D)
    return dict(shape=shape, weights=w, inputs=x, conv_state=h16(C * 3, 0.023, 0.04, 1, C, 3),
                state=state)


def workload_batched_decode(batch: int = 64, sets: int = 16, shard: int = 0) -> Dict:
    """B=64 decode, Hk=16, Hv=32, D=128, Tiled, negative-rate, bf16 inputs
    ~N(0,1), fp32 state ~N(0,0.02), conv state ~N(0,0.1); ``sets`` distinct
    per-step input sets that a long run cycles through. ``shard`` r > 0 draws
    another batch of sequences from its own seed (one per process when the
    sequences are split across processes); shard 0 is the single-process
    workload."""
    shape = Shape(16, 32, 128, map=TILED, decay=NEGATIVE_RATE, dtype="bf16")
    g = rng(SEED_BASE + 2 + 7919 * shard)
    w = layer_weights(g, shape)
    steps = [step_inputs(g, shape, batch) for _ in range(sets)]
    return dict(shape=shape, weights=w, steps=steps, batch=batch,
                conv_state=conv_state(g, shape, batch, std=0.1),
                state=delta_state(g, shape, batch, std=0.02))


def workload_multilayer_decode(layers: int = 48, batch: int = 128,
                               state_device: Optional[str] = None) -> Dict:
    """48 layers x B=128, Hk=16, Hv=48, D=128, Grouped, log-rate (A_log = ln
    U[1,16], dt_bias ~U(-0.5,0.5)), bf16 inputs ~N(0,1), fp32 states ~N(0,0.02),
    conv states ~N(0,0.1). States can be generated directly on a device (they
    total 18 GiB) with a torch generator seeded per layer."""
    shape = Shape(16, 48, 128, map=GROUPED, decay=LOG_RATE, dtype="bf16")
    g = rng(SEED_BASE + 3)
    ws = [layer_weights(g, shape) for _ in range(layers)]
    xs = [step_inputs(g, shape, batch) for _ in range(layers)]
    cs = [conv_state(g, shape, batch, std=0.1) for _ in range(layers)]
    return dict(shape=shape, weights=ws, inputs=xs, conv_states=cs, batch=batch, layers=layers)


def multilayer_state(layer: int, shape: Shape, batch: int, device: str,
                     seqs: Optional[List[int]] = None) -> torch.Tensor:
    """Layer ``layer``'s initial delta state ~N(0, 0.02), drawn per sequence
    from its own seed so a subset of sequences can be regenerated on the host."""
    idx = range(batch) if seqs is None else seqs
    out = []
    for b in idx:
        gen = torch.Generator(device="cpu").manual_seed(SEED_BASE + 3 + 1000 * (layer + 1) + b)
        out.append(torch.randn((shape.n_v_heads, shape.head_dim, shape.head_dim),
                               generator=gen, dtype=torch.float32) * 0.02)
    return torch.stack(out).to(device)


def workload_prefill(tokens: int = 4096, random_state: bool = True) -> Dict:
    """One sequence of T=4096, Hk=16, Hv=32, D=128, Grouped, log-rate, bf16
    q/k/v/z ~N(0,1), a/b ~N(0,1); initial state zero or ~N(0,0.02)."""
    shape = Shape(16, 32, 128, map=GROUPED, decay=LOG_RATE, dtype="bf16")
    g = rng(SEED_BASE + 4)
    w = layer_weights(g, shape)
    Hk, Hv, D = shape.n_k_heads, shape.n_v_heads, shape.head_dim
    q = to_dtype(normal(g, (tokens, Hk, D), 1.0), "bf16")
    k = to_dtype(normal(g, (tokens, Hk, D), 1.0), "bf16")
    v = to_dtype(normal(g, (tokens, Hv, D), 1.0), "bf16")
    z = to_dtype(normal(g, (tokens, Hv, D), 1.0), "bf16")
    a = to_dtype(normal(g, (tokens, Hv), 1.0), "bf16")
    b = to_dtype(normal(g, (tokens, Hv), 1.0), "bf16")
    s0 = delta_state(g, shape, 1, std=0.02) if random_state else torch.zeros(
        (1, Hv, D, D), dtype=torch.float32)
    return dict(shape=shape, weights=w, q=q, k=k, v=v, z=z, a=a, b=b, state=s0,
                cu_seqlens=cu_seqlens([tokens]))


def workload_varlen(n_seqs: int = 8, lo: int = 512, hi: int = 8192, decode_steps: int = 16,
                    lengths: Optional[List[int]] = None) -> Dict:
    """8 sequences of lengths U[512,8192] (seeded, as drawn) packed through
    cu_seqlens, Hk=16, Hv=64, D=128, Tiled, log-rate, bf16 inputs ~N(0,1),
    prior state ~N(0,0.02), conv state ~N(0,0.1), then ``decode_steps`` more
    tokens per sequence."""
    shape = Shape(16, 64, 128, map=TILED, decay=LOG_RATE, dtype="bf16")
    if lengths is None:
        lengths = varlen_lengths(SEED_BASE + 5, n_seqs, lo, hi)
    g = rng(SEED_BASE + 5 + 100)
    w = layer_weights(g, shape)
    total = int(sum(lengths))
    x = step_inputs(g, shape, total)
    dec = [step_inputs(g, shape, len(lengths)) for _ in range(decode_steps)]
    return dict(shape=shape, weights=w, lengths=lengths, cu_seqlens=cu_seqlens(lengths),
                inputs=x, decode=dec,
                conv_state=conv_state(g, shape, len(lengths), std=0.1),
                state=delta_state(g, shape, len(lengths), std=0.02))


def small_shape_inputs(seed: int, shape: Shape, lengths: List[int], *, state_std=0.02,
                       conv_std=0.1) -> Dict:
    """A small varlen case for parity at sizes the oracle finishes in seconds."""
    g = rng(seed)
    w = layer_weights(g, shape)
    total = int(sum(lengths))
    return dict(shape=shape, weights=w, lengths=lengths, cu_seqlens=cu_seqlens(lengths),
                inputs=step_inputs(g, shape, total),
                conv_state=conv_state(g, shape, len(lengths), std=conv_std),
                state=delta_state(g, shape, len(lengths), std=state_std))


def bytes_of(*ts: torch.Tensor) -> int:
    return int(sum(t.numel() * t.element_size() for t in ts))


def isclose_ulp_bound(dtype: str) -> float:
    """Unit roundoff of the storage dtype (half an ulp at 1.0)."""
    return {"f16": 2.0 ** -11, "bf16": 2.0 ** -8, "f32": 2.0 ** -24}[dtype]


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("annotations", "math")]
