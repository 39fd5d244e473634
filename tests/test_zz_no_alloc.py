"""gdn_prefill_chunked_static: the chunk-parallel prefill over the library's
static device scratch (no workspace argument, nothing allocated per call).
Collected last so that every other test has already exercised the library."""

import ctypes

import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
import gdn_inputs as gi
from tests.gpu_helpers import cuda

VP = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    from gated_delta_net_causal_gb300 import _build
    _build.build()
    return gdn.library()


def test_static_scratch_limit_is_checked_first(lib):
    """Sizes whose workspace exceeds the static scratch are refused on the
    host, before any pointer is looked at or any device call is made."""
    d = gdn.dims(16, 64, 128, io_dtype=torch.bfloat16)
    T = 10000
    need = gdn.gdn_prefill_workspace_size(d, 1, T)
    assert need > gdn.GDN_STATIC_SCRATCH_BYTES
    st = lib.gdn_prefill_chunked_static(ctypes.byref(d), 1, VP(0x100), T, VP(0x1000), 4096,
                                        VP(0x2000), 4096, VP(0x3000), 8192, VP(0x4000),
                                        VP(0x5000), VP(0x6000), VP(0x7000), 0, VP(0x8000),
                                        VP(0x9000), None, None, None, None)
    assert st == 2  # GDN_ERR_EXTENT
    # the 4096-token single-sequence workload fits
    assert gdn.gdn_prefill_workspace_size(gdn.dims(16, 32, 128, io_dtype=torch.bfloat16), 1,
                                          4096) <= gdn.GDN_STATIC_SCRATCH_BYTES


def _case(seed, shape, lengths):
    g = gi.rng(seed)
    Hk, Hv, D = shape.n_k_heads, shape.n_v_heads, shape.head_dim
    T = int(sum(lengths))
    w = gi.layer_weights(g, shape)
    t = lambda *s: gi.to_dtype(gi.normal(g, s, 1.0), shape.dtype)
    return (w, t(T, Hk * D), t(T, Hk * D), t(T, Hv * D), t(T, Hv, D), t(T, Hv), t(T, Hv),
            gi.delta_state(g, shape, len(lengths), std=0.02))


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_static_scratch_matches_workspace_path_bit_for_bit(dtype):
    """Same kernels, same inputs: the static-scratch call and the workspace
    call give identical outputs and states (f16 takes the single-pass kernel
    on both sides)."""
    shape = gi.Shape(2, 8, 128, map=gi.TILED, decay=gi.LOG_RATE, dtype=dtype)
    lengths = [130, 0, 63, 64, 1]
    w, q, k, v, z, a, b, S0 = _case(77, shape, lengths)
    cu = cuda(gi.cu_seqlens(lengths))
    d = gdn.dims(2, 8, 128, map=gi.TILED, io_dtype=gi.DTYPES[dtype])
    T = q.shape[0]
    args = [cuda(x) for x in (q, k, v, a, b)] + [cuda(w.decay_param), cuda(w.dt_bias)]
    res = []
    for fn in (gdn.gdn_prefill_chunked, gdn.gdn_prefill_chunked_static):
        st = cuda(S0)
        core = torch.full((T, 8, 128), float("nan"), device="cuda")
        out = torch.full((T, 8, 128), float("nan"), device="cuda", dtype=gi.DTYPES[dtype])
        fn(d, cu, *args, st, core_out=core, z=cuda(z), norm_w=cuda(w.norm_w), out=out)
        torch.cuda.synchronize()
        res.append((core.cpu(), out.cpu(), st.cpu()))
    for x, y in zip(*res):
        assert torch.equal(x, y)
    assert gdn.gdn_device_error() == 0


@pytest.mark.gpu
def test_static_scratch_serial_calls_on_one_stream():
    """Back-to-back calls on one stream reuse the scratch safely: two
    sequences prefilled by consecutive calls equal the same work in one."""
    shape = gi.Shape(1, 2, 128, dtype="bf16")
    w, q, k, v, z, a, b, S0 = _case(78, shape, [100, 100])
    d = gdn.dims(1, 2, 128)
    wargs = [cuda(w.decay_param), cuda(w.dt_bias)]
    st_one = cuda(S0)
    core_one = torch.empty((200, 2, 128), device="cuda")
    gdn.gdn_prefill_chunked_static(d, cuda(gi.cu_seqlens([100, 100])), cuda(q), cuda(k), cuda(v),
                                   cuda(a), cuda(b), *wargs, st_one, core_out=core_one)
    st_two = cuda(S0)
    core_two = torch.empty((200, 2, 128), device="cuda")
    for n in range(2):
        sl = slice(100 * n, 100 * (n + 1))
        gdn.gdn_prefill_chunked_static(d, cuda(gi.cu_seqlens([100])), cuda(q[sl]), cuda(k[sl]),
                                       cuda(v[sl]), cuda(a[sl]), cuda(b[sl]), *wargs,
                                       st_two[n:n + 1], core_out=core_two[sl])
    torch.cuda.synchronize()
    assert torch.equal(core_one.cpu(), core_two.cpu())
    assert torch.equal(st_one.cpu(), st_two.cpu())


@pytest.mark.gpu
@pytest.mark.parametrize("T", [4096, 5025])
def test_static_scratch_full_size_bit_for_bit(T):
    """The 4096-token single-sequence workload (Hk=16, Hv=32, bf16, fused
    norm) and the longest sequence whose workspace still fits the static
    scratch (5,025 tokens, within 2 % of its size): the static-scratch call
    equals the workspace call bit for bit, so the scratch's far end (the
    carry's core-output region) is addressed the same way."""
    wl = gi.workload_prefill(T, random_state=True)
    shape, w = wl["shape"], wl["weights"]
    d = gdn.dims(16, 32, 128, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    need = gdn.gdn_prefill_workspace_size(d, 1, T)
    assert need <= gdn.GDN_STATIC_SCRATCH_BYTES
    if T == 5025:
        assert need > 0.98 * gdn.GDN_STATIC_SCRATCH_BYTES
        assert gdn.gdn_prefill_workspace_size(d, 1, T + 1) > gdn.GDN_STATIC_SCRATCH_BYTES
    cu = cuda(wl["cu_seqlens"])
    q, k, v = (cuda(wl[n]).reshape(T, -1) for n in ("q", "k", "v"))
    a, b, z = cuda(wl["a"]), cuda(wl["b"]), cuda(wl["z"])
    args = [cuda(w.decay_param), cuda(w.dt_bias)]
    res = []
    for fn in (gdn.gdn_prefill_chunked, gdn.gdn_prefill_chunked_static):
        st = cuda(wl["state"])
        out = torch.full((T, 32, 128), float("nan"), device="cuda", dtype=torch.bfloat16)
        fn(d, cu, q, k, v, a, b, *args, st, z=z, norm_w=cuda(w.norm_w), out=out)
        torch.cuda.synchronize()
        res.append((out.cpu(), st.cpu()))
    for x, y in zip(*res):
        assert torch.equal(x, y)
    assert not torch.isnan(res[0][0].float()).any()
    assert gdn.gdn_device_error() == 0
