"""GPU parity of gdn_conv_update and gdn_gated_rmsnorm against the oracle."""

import numpy as np
import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
import gdn_inputs as gi
import oracle
from tests.gpu_helpers import F64, assert_lowp, cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("lengths", [[5], [0, 1, 2, 3, 4, 64, 100, 0, 7], [1] * 9,
                                     [300, 1, 65]])
def test_conv_update_varlen(dtype, lengths):
    shape = gi.Shape(2, 4, 64, dtype=dtype)
    data = gi.small_shape_inputs(40 + len(lengths), shape, lengths)
    x, w, cs = data["inputs"].mixed_qkv, data["weights"].conv_w, data["conv_state"]
    cu = data["cu_seqlens"]
    d = gdn.dims(2, 4, 64, io_dtype=gi.DTYPES[dtype])
    xs, csd = cuda(x), cuda(cs)
    y = torch.full_like(xs, float("nan"))
    gdn.gdn_conv_update(d, cuda(cu), xs, cuda(w), csd, y)
    torch.cuda.synchronize()
    ry, rcs = oracle.conv_varlen(F64(x), F64(w), F64(cs), cu.numpy())
    assert np.array_equal(F64(csd.cpu()), rcs), "conv state must be a bit copy"
    if x.shape[0]:
        assert_lowp(y.cpu(), ry, dtype, f"conv y {lengths}", rel=1e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("hk,hv,D", [(1, 1, 32), (1, 3, 64)])
def test_conv_update_partial_channel_tile(dtype, hk, hv, D):
    """Channel counts (96, 320) that leave the last 512-byte channel tile
    partly empty, with sequences crossing the 64-token tiles."""
    shape = gi.Shape(hk, hv, D, dtype=dtype)
    lengths = [70, 3, 0, 130, 1]
    data = gi.small_shape_inputs(50 + D + hv, shape, lengths)
    x, w, cs = data["inputs"].mixed_qkv, data["weights"].conv_w, data["conv_state"]
    d = gdn.dims(hk, hv, D, io_dtype=gi.DTYPES[dtype])
    xs, csd = cuda(x), cuda(cs)
    y = torch.full_like(xs, float("nan"))
    gdn.gdn_conv_update(d, cuda(data["cu_seqlens"]), xs, cuda(w), csd, y)
    torch.cuda.synchronize()
    ry, rcs = oracle.conv_varlen(F64(x), F64(w), F64(cs), data["cu_seqlens"].numpy())
    assert np.array_equal(F64(csd.cpu()), rcs), "conv state must be a bit copy"
    assert_lowp(y.cpu(), ry, dtype, f"conv y C={(2 * hk + hv) * D}", rel=1e-5)


def test_conv_update_large_batch_tail_tiles():
    """Many sequences and a token count that is not a multiple of the tile."""
    shape = gi.Shape(4, 8, 128, dtype="bf16")
    lengths = [int(v) for v in gi.rng(9).integers(0, 40, size=37)]
    data = gi.small_shape_inputs(41, shape, lengths)
    x, w, cs = data["inputs"].mixed_qkv, data["weights"].conv_w, data["conv_state"]
    d = gdn.dims(4, 8, 128)
    xs, csd = cuda(x), cuda(cs)
    y = torch.empty_like(xs)
    gdn.gdn_conv_update(d, cuda(data["cu_seqlens"]), xs, cuda(w), csd, y)
    torch.cuda.synchronize()
    ry, rcs = oracle.conv_varlen(F64(x), F64(w), F64(cs), data["cu_seqlens"].numpy())
    assert np.array_equal(F64(csd.cpu()), rcs)
    assert_lowp(y.cpu(), ry, "bf16", "conv y", rel=1e-5)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("D", [32, 64, 96, 128])
def test_gated_rmsnorm(dtype, D):
    g = gi.rng(D)
    rows = 1000 + D
    o = gi.to_dtype(gi.normal(g, (rows, D), 0.3), "f32")
    o[3] = 0.0  # an all-zero row: output zero, no NaN
    z = gi.to_dtype(gi.normal(g, (rows, D), 1.0), dtype)
    w = gi.to_dtype(0.82 + 0.013 * np.arange(D), "f32")
    d = gdn.dims(1, 1, D, io_dtype=gi.DTYPES[dtype])
    y = torch.full((rows, D), float("nan"), device="cuda", dtype=gi.DTYPES[dtype])
    gdn.gdn_gated_rmsnorm(d, cuda(o), cuda(z), cuda(w), y)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(F64(o), F64(z), F64(w), 1e-6)
    assert_lowp(y.cpu(), ref, dtype, f"gated rmsnorm D={D}")
