"""GB300 gated delta-net core: a thin Python binding over libgdn.so.

Each function takes torch CUDA tensors, checks only what marshalling needs
(device, dtype, contiguity, and that every tensor holds the elements the call
touches, since the C ABI sees only pointers), and calls the C-ABI entry point
of the same name on the current torch CUDA stream. Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback. If libgdn.so is
missing the import of the library raises.

The C ABI itself is declared in ``include/gdn.h``.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

GDN_OK = 0
GDN_MAP_GROUPED, GDN_MAP_TILED = 0, 1
GDN_DECAY_LOG_RATE, GDN_DECAY_NEGATIVE_RATE = 0, 1
GDN_F16, GDN_BF16, GDN_F32 = 0, 1, 2
GDN_QK_PRENORMALIZED, GDN_GATES_PRECOMPUTED, GDN_PREFILL_CUDA_CORES = 1, 2, 4
GDN_PREFILL_CARRY_WHOLE, GDN_PREFILL_CARRY_SLICED = 8, 16

_TORCH_TO_GDN = {torch.float16: GDN_F16, torch.bfloat16: GDN_BF16, torch.float32: GDN_F32}
_GDN_TO_TORCH = {v: k for k, v in _TORCH_TO_GDN.items()}


class GdnDims(ctypes.Structure):
    _fields_ = [("n_k_heads", ctypes.c_int32), ("n_v_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("map", ctypes.c_int32),
                ("decay", ctypes.c_int32), ("io_dtype", ctypes.c_int32),
                ("l2_eps", ctypes.c_float), ("rms_eps", ctypes.c_float)]


def dims(n_k_heads: int, n_v_heads: int, head_dim: int, map: int = GDN_MAP_GROUPED,
         decay: int = GDN_DECAY_LOG_RATE, io_dtype=torch.bfloat16, l2_eps: float = 1e-6,
         rms_eps: float = 1e-6) -> GdnDims:
    dt = _TORCH_TO_GDN[io_dtype] if isinstance(io_dtype, torch.dtype) else int(io_dtype)
    return GdnDims(n_k_heads, n_v_heads, head_dim, map, decay, dt, l2_eps, rms_eps)


class GdnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


_lib = None
LIB_PATH = _build.LIB


def library() -> ctypes.CDLL:
    """Load libgdn.so (built by ``__graft_entry__.build()`` / ``_build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                              "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        pd = ctypes.POINTER(GdnDims)
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_status_string.argtypes = [i32]
        L.gdn_version.restype = i32
        L.gdn_version.argtypes = []
        L.gdn_host_pointer.restype = ctypes.c_int
        L.gdn_host_pointer.argtypes = [vp, ctypes.POINTER(vp)]
        L.gdn_qkv_features.restype = i64
        L.gdn_qkv_features.argtypes = [pd]
        L.gdn_conv_update.restype = ctypes.c_int
        L.gdn_conv_update.argtypes = [pd, i32, vp, i64, vp, vp, vp, vp, vp]
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [pd, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.gdn_decode_multi.restype = ctypes.c_int
        L.gdn_decode_multi.argtypes = [pd, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                       vp, vp]
        L.gdn_decode_step_slots.restype = ctypes.c_int
        L.gdn_decode_step_slots.argtypes = [pd, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                            vp, vp, vp, vp]
        L.gdn_prefill_chunked.restype = ctypes.c_int
        L.gdn_prefill_chunked.argtypes = [pd, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, vp, vp,
                                          vp, i32, vp, vp, vp, vp, vp, vp, i64, vp]
        L.gdn_prefill_chunked_static.restype = ctypes.c_int
        L.gdn_prefill_chunked_static.argtypes = [pd, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp,
                                                 vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]
        L.gdn_prefill_workspace_size.restype = ctypes.c_int
        L.gdn_prefill_workspace_size.argtypes = [pd, i32, i64, i32, ctypes.POINTER(i64)]
        L.gdn_gated_rmsnorm.restype = ctypes.c_int
        L.gdn_gated_rmsnorm.argtypes = [pd, i64, vp, vp, vp, vp, vp]
        L.gdn_device_error.restype = ctypes.c_int
        L.gdn_device_error.argtypes = [ctypes.POINTER(i32), i32]
        L.gdn_selftest_wait_timeout.restype = ctypes.c_int
        L.gdn_selftest_wait_timeout.argtypes = [i64, vp, vp]
        L.gdn_linear.restype = ctypes.c_int
        L.gdn_linear.argtypes = [i32, i32, i32, vp, i64, vp, vp, vp, i64, vp, i64, vp]
        L.gdn_linear_workspace_size.restype = ctypes.c_int
        L.gdn_linear_workspace_size.argtypes = [i32, i32, i32, ctypes.POINTER(i64)]
        L.gdn_decode_layer.restype = ctypes.c_int
        L.gdn_decode_layer.argtypes = [pd, i32, i32, vp, ctypes.POINTER(GdnLayerWeights), vp, vp, vp, vp,
                                       i64, vp]
        L.gdn_decode_layer_workspace_size.restype = ctypes.c_int
        L.gdn_decode_layer_workspace_size.argtypes = [pd, i32, i32, ctypes.POINTER(i64)]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return library().gdn_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != GDN_OK:
        raise GdnError(status, f"{what}: {status_string(status)}")


def gdn_host_pointer(t: torch.Tensor) -> int:
    """The device address of a pinned host tensor's data (gdn_host_pointer)."""
    dev = ctypes.c_void_p()
    _check(library().gdn_host_pointer(ctypes.c_void_p(t.data_ptr()), ctypes.byref(dev)),
           "gdn_host_pointer")
    return int(dev.value)


def _ptr(t: Optional[torch.Tensor], name: str, dtype=None, host_ok: bool = False) -> Optional[int]:
    """A tensor argument's device address. With host_ok a pinned host tensor
    is accepted too and passed as its mapped device address (the kernel then
    reads or writes it over the host link)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda and not (host_ok and t.device.type == "cpu" and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if host_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr() if t.is_cuda else gdn_host_pointer(t)


def _shape(d: GdnDims):
    Hk, Hv, D = d.n_k_heads, d.n_v_heads, d.head_dim
    return Hk, Hv, D, (2 * Hk + Hv) * D


def _need(t, name: str, n: int):
    """The C ABI sees only pointers: a tensor handed to a call must hold at
    least the elements the call touches, or a kernel would read or write past
    it. Checked here, before anything reaches the library."""
    if isinstance(t, torch.Tensor) and t.numel() < n:
        raise ValueError(f"{name} holds {t.numel()} elements; the call uses {n}")


def _need_rows(t, name: str, rows: int, width: int):
    """A token-strided operand: at least `rows` rows, each `width` contiguous
    elements from the row's start."""
    if t.dim() < 2 or t.shape[0] < rows:
        raise ValueError(f"{name} must have at least {rows} rows")
    if rows > 0 and (not t[0].is_contiguous() or t[0].numel() < width):
        raise ValueError(f"{name}: each row must hold {width} contiguous elements")


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _io(d: GdnDims):
    return _GDN_TO_TORCH[d.io_dtype]


def gdn_conv_update(d: GdnDims, cu_seqlens: torch.Tensor, x: torch.Tensor, conv_w: torch.Tensor,
                    conv_state: torch.Tensor, y: torch.Tensor, stream=None) -> torch.Tensor:
    io = _io(d)
    n = cu_seqlens.numel() - 1
    total = x.shape[0] if x.dim() > 0 else 0
    _, _, _, C = _shape(d)
    for t, name, cnt in ((x, "x", total * C), (y, "y", total * C), (conv_w, "conv_w", C * 4),
                         (conv_state, "conv_state", max(n, 0) * C * 3)):
        _need(t, name, cnt)
    _check(library().gdn_conv_update(
        ctypes.byref(d), n, _ptr(cu_seqlens, "cu_seqlens", torch.int32), total,
        _ptr(x, "x", io), _ptr(conv_w, "conv_w", io), _ptr(conv_state, "conv_state", io),
        _ptr(y, "y", io), _stream(stream)), "gdn_conv_update")
    return y


def _check_decode_sizes(d, batch, tokens, slots, mixed_qkv, a, b, decay_param, dt_bias, conv_w,
                        conv_state, state, core_out, z, norm_w, out):
    _, Hv, D, C = _shape(d)
    rows = batch * tokens
    for t, name, cnt in ((mixed_qkv, "mixed_qkv", rows * C), (a, "a", rows * Hv),
                         (b, "b", rows * Hv), (decay_param, "decay_param", Hv),
                         (dt_bias, "dt_bias", Hv), (conv_w, "conv_w", C * 4),
                         (conv_state, "conv_state", slots * C * 3),
                         (state, "state", slots * Hv * D * D),
                         (core_out, "core_out", rows * Hv * D), (z, "z", rows * Hv * D),
                         (norm_w, "norm_w", D), (out, "out", rows * Hv * D)):
        _need(t, name, cnt)


def gdn_decode_step(d: GdnDims, mixed_qkv, a, b, decay_param, dt_bias, conv_w, conv_state,
                    state, core_out=None, z=None, norm_w=None, out=None, stream=None):
    """mixed_qkv, a, b, z, core_out and out may be pinned host tensors: the
    kernel reads and writes them in place over the host link."""
    io = _io(d)
    batch = mixed_qkv.shape[0]
    _check_decode_sizes(d, batch, 1, batch, mixed_qkv, a, b, decay_param, dt_bias, conv_w,
                        conv_state, state, core_out, z, norm_w, out)
    f32 = torch.float32
    _check(library().gdn_decode_step(
        ctypes.byref(d), batch, _ptr(mixed_qkv, "mixed_qkv", io, True), _ptr(a, "a", io, True),
        _ptr(b, "b", io, True), _ptr(decay_param, "decay_param", f32),
        _ptr(dt_bias, "dt_bias", f32), _ptr(conv_w, "conv_w", io),
        _ptr(conv_state, "conv_state", io), _ptr(state, "state", f32),
        _ptr(core_out, "core_out", f32, True), _ptr(z, "z", io, True),
        _ptr(norm_w, "norm_w", f32), _ptr(out, "out", io, True), _stream(stream)),
        "gdn_decode_step")
    return core_out, out


def gdn_decode_multi(d: GdnDims, mixed_qkv, a, b, decay_param, dt_bias, conv_w, conv_state,
                     state, core_out=None, z=None, norm_w=None, out=None, stream=None):
    """T consecutive tokens per sequence: mixed_qkv [B][T][C], a and b
    [B][T][Hv], z / core_out / out [B][T][Hv][D]."""
    io = _io(d)
    if mixed_qkv.dim() != 3:
        raise ValueError("mixed_qkv must be [B][T][C]")
    batch, tokens = mixed_qkv.shape[0], mixed_qkv.shape[1]
    _check_decode_sizes(d, batch, tokens, batch, mixed_qkv, a, b, decay_param, dt_bias, conv_w,
                        conv_state, state, core_out, z, norm_w, out)
    f32 = torch.float32
    _check(library().gdn_decode_multi(
        ctypes.byref(d), batch, tokens, _ptr(mixed_qkv, "mixed_qkv", io), _ptr(a, "a", io),
        _ptr(b, "b", io), _ptr(decay_param, "decay_param", f32), _ptr(dt_bias, "dt_bias", f32),
        _ptr(conv_w, "conv_w", io), _ptr(conv_state, "conv_state", io),
        _ptr(state, "state", f32), _ptr(core_out, "core_out", f32), _ptr(z, "z", io),
        _ptr(norm_w, "norm_w", f32), _ptr(out, "out", io), _stream(stream)), "gdn_decode_multi")
    return core_out, out


def gdn_decode_step_slots(d: GdnDims, state_slots, mixed_qkv, a, b, decay_param, dt_bias, conv_w,
                          conv_state, state, core_out=None, z=None, norm_w=None, out=None,
                          stream=None):
    """gdn_decode_step where batch row b works on state[state_slots[b]] and
    conv_state[state_slots[b]] of a pool (state [P][Hv][D][D], conv_state
    [P][C][3]); a negative slot marks a padded row."""
    io = _io(d)
    batch = mixed_qkv.shape[0]
    if state_slots.numel() != batch:
        raise ValueError("state_slots must hold one entry per batch row")
    if conv_state.shape[0] != state.shape[0]:
        raise ValueError("state and conv_state must hold the same number of slots")
    _check_decode_sizes(d, batch, 1, state.shape[0], mixed_qkv, a, b, decay_param, dt_bias,
                        conv_w, conv_state, state, core_out, z, norm_w, out)
    f32 = torch.float32
    _check(library().gdn_decode_step_slots(
        ctypes.byref(d), batch, _ptr(state_slots, "state_slots", torch.int32), state.shape[0],
        _ptr(mixed_qkv, "mixed_qkv", io), _ptr(a, "a", io), _ptr(b, "b", io),
        _ptr(decay_param, "decay_param", f32), _ptr(dt_bias, "dt_bias", f32),
        _ptr(conv_w, "conv_w", io), _ptr(conv_state, "conv_state", io),
        _ptr(state, "state", f32), _ptr(core_out, "core_out", f32), _ptr(z, "z", io),
        _ptr(norm_w, "norm_w", f32), _ptr(out, "out", io), _stream(stream)),
        "gdn_decode_step_slots")
    return core_out, out


def _token_stride(t: torch.Tensor, name: str) -> int:
    if t.dim() < 2 or t.stride(-1) != 1:
        raise ValueError(f"{name} must have a unit innermost stride")
    return int(t.stride(0))


def _base_ptr(t: torch.Tensor, name: str, dtype) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def gdn_prefill_workspace_size(d: GdnDims, num_seqs: int, total_tokens: int,
                               flags: int = 0) -> int:
    n = ctypes.c_int64(0)
    _check(library().gdn_prefill_workspace_size(ctypes.byref(d), int(num_seqs), int(total_tokens),
                                                int(flags), ctypes.byref(n)),
           "gdn_prefill_workspace_size")
    return n.value


def _check_prefill_sizes(d, cu_seqlens, q, k, v, a, b, decay_param, dt_bias, state, core_out, z,
                         norm_w, out):
    Hk, Hv, D, _ = _shape(d)
    T, n = q.shape[0], max(cu_seqlens.numel() - 1, 0)
    _need_rows(q, "q", T, Hk * D)
    _need_rows(k, "k", T, Hk * D)
    _need_rows(v, "v", T, Hv * D)
    for t, name, cnt in ((a, "a", T * Hv), (b, "b", T * Hv), (decay_param, "decay_param", Hv),
                         (dt_bias, "dt_bias", Hv), (state, "state", n * Hv * D * D),
                         (core_out, "core_out", T * Hv * D), (z, "z", T * Hv * D),
                         (norm_w, "norm_w", D), (out, "out", T * Hv * D)):
        _need(t, name, cnt)


def gdn_prefill_chunked(d: GdnDims, cu_seqlens, q, k, v, a, b, decay_param, dt_bias, state,
                        core_out=None, z=None, norm_w=None, out=None, flags: int = 0,
                        workspace="auto", stream=None):
    """q, k: [T][Hk*D] (or views with a token stride, e.g. column slices of the
    conv output); v: [T][Hv*D] likewise. With GDN_GATES_PRECOMPUTED a and b are
    fp32 g and beta.

    workspace: "auto" allocates the scratch the library asks for (a torch
    CUDA byte tensor, only when a workspace path applies); None passes no
    workspace (the single-pass kernels); or a CUDA uint8 tensor of at least
    gdn_prefill_workspace_size bytes."""
    io = _io(d)
    f32 = torch.float32
    gate_dt = f32 if (flags & GDN_GATES_PRECOMPUTED) else io
    _check_prefill_sizes(d, cu_seqlens, q, k, v, a, b, decay_param, dt_bias, state, core_out, z,
                         norm_w, out)
    total = q.shape[0]
    n = cu_seqlens.numel() - 1
    ws_ptr, ws_bytes = None, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace must be 'auto', None or a CUDA tensor")
        need = gdn_prefill_workspace_size(d, n, total, flags)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
            if isinstance(stream, torch.cuda.Stream):
                # freed when this call returns: keep it from being reused
                # before the kernels on that stream are done with it
                workspace.record_stream(stream)
        else:
            workspace = None
    if workspace is not None:
        ws_ptr = _ptr(workspace, "workspace", torch.uint8)
        ws_bytes = workspace.numel()
    _check(library().gdn_prefill_chunked(
        ctypes.byref(d), n, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
        total, _base_ptr(q, "q", io), _token_stride(q, "q"), _base_ptr(k, "k", io),
        _token_stride(k, "k"), _base_ptr(v, "v", io), _token_stride(v, "v"),
        _ptr(a, "a", gate_dt), _ptr(b, "b", gate_dt), _ptr(decay_param, "decay_param", f32),
        _ptr(dt_bias, "dt_bias", f32), int(flags), _ptr(state, "state", f32),
        _ptr(core_out, "core_out", f32), _ptr(z, "z", io), _ptr(norm_w, "norm_w", f32),
        _ptr(out, "out", io), ws_ptr, ws_bytes, _stream(stream)), "gdn_prefill_chunked")
    return core_out, out


GDN_STATIC_SCRATCH_BYTES = 160 << 20


def gdn_prefill_chunked_static(d: GdnDims, cu_seqlens, q, k, v, a, b, decay_param, dt_bias,
                               state, core_out=None, z=None, norm_w=None, out=None,
                               flags: int = 0, stream=None):
    """gdn_prefill_chunked over the library's static device scratch (no
    workspace, no allocation). Calls must not overlap in time on one device."""
    io = _io(d)
    f32 = torch.float32
    gate_dt = f32 if (flags & GDN_GATES_PRECOMPUTED) else io
    _check_prefill_sizes(d, cu_seqlens, q, k, v, a, b, decay_param, dt_bias, state, core_out, z,
                         norm_w, out)
    _check(library().gdn_prefill_chunked_static(
        ctypes.byref(d), cu_seqlens.numel() - 1, _ptr(cu_seqlens, "cu_seqlens", torch.int32),
        q.shape[0], _base_ptr(q, "q", io), _token_stride(q, "q"), _base_ptr(k, "k", io),
        _token_stride(k, "k"), _base_ptr(v, "v", io), _token_stride(v, "v"),
        _ptr(a, "a", gate_dt), _ptr(b, "b", gate_dt), _ptr(decay_param, "decay_param", f32),
        _ptr(dt_bias, "dt_bias", f32), int(flags), _ptr(state, "state", f32),
        _ptr(core_out, "core_out", f32), _ptr(z, "z", io), _ptr(norm_w, "norm_w", f32),
        _ptr(out, "out", io), _stream(stream)), "gdn_prefill_chunked_static")
    return core_out, out


def gdn_gated_rmsnorm(d: GdnDims, o, z, norm_w, y, stream=None):
    io = _io(d)
    rows = o.numel() // d.head_dim
    for t, name in ((z, "z"), (y, "y")):
        _need(t, name, rows * d.head_dim)
    _need(norm_w, "norm_w", d.head_dim)
    _check(library().gdn_gated_rmsnorm(
        ctypes.byref(d), rows, _ptr(o, "o", torch.float32), _ptr(z, "z", io),
        _ptr(norm_w, "norm_w", torch.float32), _ptr(y, "y", io), _stream(stream)),
        "gdn_gated_rmsnorm")
    return y


def gdn_device_error(clear: bool = True) -> int:
    st = ctypes.c_int32(0)
    _check(library().gdn_device_error(ctypes.byref(st), 1 if clear else 0), "gdn_device_error")
    return st.value


class GdnLayerWeights(ctypes.Structure):
    """gdn_layer_weights: device pointers of one layer's weights."""
    _fields_ = [("w_in", ctypes.c_void_p), ("b_in", ctypes.c_void_p), ("w_out", ctypes.c_void_p),
                ("b_out", ctypes.c_void_p), ("conv_w", ctypes.c_void_p), ("decay_param", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("norm_w", ctypes.c_void_p)]


def gdn_linear_workspace_size(M: int, N: int, K: int) -> int:
    n = ctypes.c_int64(0)
    _check(library().gdn_linear_workspace_size(int(M), int(N), int(K), ctypes.byref(n)),
           "gdn_linear_workspace_size")
    return n.value


def gdn_linear(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, bias: Optional[torch.Tensor] = None,
               workspace="auto", stream=None) -> torch.Tensor:
    """y[M][N] = x[M][K] w[N][K]^T (+ bias), bf16 (rows of x and y may be
    strided)."""
    bf = torch.bfloat16
    if x.dim() != 2 or w.dim() != 2 or y.dim() != 2:
        raise ValueError("x, w and y must be 2-D")
    M, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or y.shape[0] != M or y.shape[1] != N:
        raise ValueError(f"shapes: x {tuple(x.shape)}, w {tuple(w.shape)}, y {tuple(y.shape)}")
    for t, name in ((x, "x"), (y, "y")):
        if t.dtype != bf or not t.is_cuda or t.stride(1) != 1:
            raise ValueError(f"{name} must be a CUDA bf16 tensor with unit column stride")
    _need(bias, "bias", N)
    need = gdn_linear_workspace_size(M, N, K)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device) if need > 0 else None
    _need(workspace, "workspace", need)
    ws_ptr = _ptr(workspace, "workspace", torch.uint8) if workspace is not None else None
    _check(library().gdn_linear(int(M), int(N), int(K), x.data_ptr(), int(x.stride(0)), _ptr(w, "w", bf),
                                _ptr(bias, "bias", torch.float32), y.data_ptr(), int(y.stride(0)),
                                ws_ptr, int(workspace.numel()) if workspace is not None else 0,
                                _stream(stream)), "gdn_linear")
    return y


def gdn_decode_layer_workspace_size(d: GdnDims, hidden: int, batch: int) -> int:
    n = ctypes.c_int64(0)
    _check(library().gdn_decode_layer_workspace_size(ctypes.byref(d), int(hidden), int(batch),
                                                     ctypes.byref(n)), "gdn_decode_layer_workspace_size")
    return n.value


def gdn_decode_layer(d: GdnDims, x: torch.Tensor, w_in, w_out, conv_w, decay_param, dt_bias, norm_w,
                     conv_state, state, y, b_in=None, b_out=None, workspace="auto", stream=None):
    """One decode step of a whole layer: x [batch][hidden] -> y [batch][hidden]
    (bf16), conv_state and state updated in place."""
    bf, f32 = torch.bfloat16, torch.float32
    Hk, Hv, D, C = _shape(d)
    batch, hidden = x.shape
    n_in = (C + Hv * D + 2 * Hv + 63) // 64 * 64
    _need(w_in, "w_in", n_in * hidden)
    _need(b_in, "b_in", n_in)
    _need(w_out, "w_out", hidden * Hv * D)
    _need(b_out, "b_out", hidden)
    _need(conv_w, "conv_w", C * 4)
    for t, name in ((decay_param, "decay_param"), (dt_bias, "dt_bias")):
        _need(t, name, Hv)
    _need(norm_w, "norm_w", D)
    _need(conv_state, "conv_state", batch * C * 3)
    _need(state, "state", batch * Hv * D * D)
    _need(y, "y", batch * hidden)
    need = gdn_decode_layer_workspace_size(d, hidden, batch)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    _need(workspace, "workspace", need)
    wts = GdnLayerWeights(_ptr(w_in, "w_in", bf), _ptr(b_in, "b_in", f32), _ptr(w_out, "w_out", bf),
                          _ptr(b_out, "b_out", f32), _ptr(conv_w, "conv_w", bf),
                          _ptr(decay_param, "decay_param", f32), _ptr(dt_bias, "dt_bias", f32),
                          _ptr(norm_w, "norm_w", f32))
    _check(library().gdn_decode_layer(ctypes.byref(d), int(hidden), int(batch), _ptr(x, "x", bf),
                                      ctypes.byref(wts), _ptr(conv_state, "conv_state", bf),
                                      _ptr(state, "state", f32), _ptr(y, "y", bf),
                                      _ptr(workspace, "workspace", torch.uint8), int(workspace.numel()),
                                      _stream(stream)), "gdn_decode_layer")
    return y


def gdn_selftest_wait_timeout(limit_ns: int, gave_up: torch.Tensor, stream=None):
    """A device-side bounded wait made to give up after limit_ns; gave_up is a
    CUDA int32 tensor of one element, set to 1 by the kernel."""
    if gave_up.numel() != 1:
        raise ValueError("gave_up must have one element")
    _check(library().gdn_selftest_wait_timeout(int(limit_ns), _ptr(gave_up, "gave_up", torch.int32),
                                               _stream(stream)), "gdn_selftest_wait_timeout")


def gdn_qkv_features(d: GdnDims) -> int:
    return int(library().gdn_qkv_features(ctypes.byref(d)))


def gdn_version() -> int:
    return int(library().gdn_version())


__all__ = ["GdnDims", "GdnError", "dims", "library", "status_string", "gdn_conv_update",
           "gdn_decode_step", "gdn_decode_multi", "gdn_decode_step_slots", "gdn_prefill_chunked", "gdn_prefill_workspace_size",
           "gdn_prefill_chunked_static", "GDN_STATIC_SCRATCH_BYTES", "gdn_gated_rmsnorm", "gdn_device_error",
           "gdn_selftest_wait_timeout", "gdn_linear", "gdn_linear_workspace_size", "gdn_decode_layer",
           "gdn_decode_layer_workspace_size", "GdnLayerWeights",
           "gdn_qkv_features", "gdn_version", "gdn_host_pointer", "GDN_MAP_GROUPED", "GDN_MAP_TILED",
           "GDN_DECAY_LOG_RATE", "GDN_DECAY_NEGATIVE_RATE", "GDN_F16", "GDN_BF16", "GDN_F32",
           "GDN_QK_PRENORMALIZED", "GDN_GATES_PRECOMPUTED", "GDN_PREFILL_CUDA_CORES",
           "GDN_PREFILL_CARRY_WHOLE", "GDN_PREFILL_CARRY_SLICED", "LIB_PATH"]
