"""The device-side give-up path of the bounded waits, made to run out on
purpose (an mbarrier that nothing arrives on, no copy or MMA in flight): the
kernel records GDN_ERR_TIMEOUT, exits after about its limit, and the context
stays usable for the next call."""

import time

import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
import gdn_inputs as gi
import oracle
from tests.gpu_helpers import F64, assert_lowp, cuda

GDN_ERR_TIMEOUT = 7


@pytest.mark.gpu
@pytest.mark.parametrize("limit_ms", [1, 20])
def test_bounded_wait_gives_up_with_timeout_status(limit_ms):
    gdn.gdn_device_error(clear=True)
    gave_up = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    gdn.gdn_selftest_wait_timeout(limit_ms * 1_000_000, gave_up)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(gave_up.item()) == 1
    assert gdn.gdn_device_error(clear=True) == GDN_ERR_TIMEOUT
    assert gdn.gdn_device_error() == 0  # cleared
    # it waited about its limit, not the library's usual 2 s
    assert limit_ms * 1e-3 <= elapsed < limit_ms * 1e-3 + 1.0

    # the context is usable: a gated norm right after gives the oracle's rows
    d = gdn.dims(2, 4, 128, io_dtype=torch.bfloat16)
    g = gi.rng(4242)
    o = torch.from_numpy(gi.normal(g, (16, 128), 1.0).astype("float32"))
    z = gi.to_dtype(gi.normal(g, (16, 128), 1.0), "bf16")
    nw = torch.from_numpy(gi.normal(g, (128,), 1.0).astype("float32"))
    y = torch.empty((16, 128), device="cuda", dtype=torch.bfloat16)
    gdn.gdn_gated_rmsnorm(d, cuda(o), cuda(z), cuda(nw), y)
    torch.cuda.synchronize()
    ry = oracle.gated_rmsnorm(F64(o), F64(z), F64(nw), d.rms_eps)
    assert_lowp(y.cpu(), ry, "bf16", "gated norm after the timeout")
    assert gdn.gdn_device_error() == 0
