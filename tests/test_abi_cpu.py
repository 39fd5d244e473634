"""Host-side checks of the C-ABI library that need no GPU: it loads, exports
every function include/gdn.h declares, and rejects bad arguments on the host
before anything is launched."""

import ctypes
import os
import re

import pytest
import torch

import gated_delta_net_causal_gb300 as gdn
from gated_delta_net_causal_gb300 import _build
from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "gdn.h")

# fake device addresses are only safe where no launch can happen at all
no_device = pytest.mark.skipif(torch.cuda.is_available(),
                               reason="fake-pointer validation runs only without a GPU")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return gdn.library()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z_]+)\s*\(", src)))


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ("gdn_conv_update", "gdn_decode_step", "gdn_prefill_chunked", "gdn_gated_rmsnorm"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    for s in range(8):
        assert gdn.status_string(s).startswith("GDN_")
    assert gdn.status_string(99) == "GDN_ERR_UNKNOWN"
    assert gdn.gdn_version() >= 300  # the release with the multi-token and slot calls


def test_prefill_workspace_size(lib):
    d = gdn.dims(16, 32, 128, io_dtype=torch.bfloat16)
    # (T + 63 N) / 64 chunk slots x (Hv x 25 KB + Hk x 16 KB), after the 1 KB index
    per_slot = 32 * 25600 + 16 * 16384
    # one sequence (Hv N <= 64): plus the sliced carry's fp32 core output
    assert gdn.gdn_prefill_workspace_size(d, 1, 4096) == 1024 + 64 * per_slot + 4096 * 32 * 512
    assert gdn.gdn_prefill_workspace_size(d, 8, 34482) == 1024 + (34482 + 63 * 8) // 64 * per_slot
    assert gdn.gdn_prefill_workspace_size(d, 1, 0) == 0
    assert gdn.gdn_prefill_workspace_size(d, 1, 4096, gdn.GDN_PREFILL_CUDA_CORES) == 0
    assert gdn.gdn_prefill_workspace_size(gdn.dims(16, 32, 64, io_dtype=torch.bfloat16), 1,
                                          4096) == 0
    assert gdn.gdn_prefill_workspace_size(gdn.dims(16, 32, 128, io_dtype=torch.float16), 1,
                                          4096) == 0
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_workspace_size(d, -1, 10)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_workspace_size(d, 1, 10, 64)  # unknown flag
    # the carry choice does not change the workspace; both at once is refused
    for carry in (gdn.GDN_PREFILL_CARRY_WHOLE, gdn.GDN_PREFILL_CARRY_SLICED):
        assert gdn.gdn_prefill_workspace_size(d, 1, 4096, carry) == 1024 + 64 * per_slot + 4096 * 32 * 512
    with pytest.raises(gdn.GdnError):
        gdn.gdn_prefill_workspace_size(d, 1, 10, gdn.GDN_PREFILL_CARRY_WHOLE | gdn.GDN_PREFILL_CARRY_SLICED)


def test_qkv_features(lib):
    assert gdn.gdn_qkv_features(gdn.dims(16, 32, 128)) == 8192
    assert gdn.gdn_qkv_features(gdn.dims(16, 48, 128)) == 10240
    assert gdn.gdn_qkv_features(gdn.dims(16, 64, 128)) == 12288
    assert gdn.gdn_qkv_features(gdn.dims(3, 4, 128)) == -1  # Hv not a multiple of Hk


VP = ctypes.c_void_p


def _decode(lib, d, batch=1, ptrs=None, core=True):
    p = dict(x=0x10000, a=0x20000, b=0x30000, dp=0x40000, dt=0x50000, w=0x60000,
             cs=0x1000000, st=0x10000000, core=0x70000000 if core else None, z=None, nw=None,
             out=None)
    if ptrs:
        p.update(ptrs)
    return lib.gdn_decode_step(ctypes.byref(d) if d is not None else None, batch,
                               *[VP(p[k]) if p[k] is not None else None for k in
                                 ("x", "a", "b", "dp", "dt", "w", "cs", "st", "core", "z", "nw",
                                  "out")], None)


@no_device
def test_decode_rejects_bad_arguments(lib):
    ok = gdn.dims(16, 32, 128)
    assert _decode(lib, None) == 1  # no dims
    assert _decode(lib, gdn.dims(3, 4, 128)) == 1  # Hv % Hk
    assert _decode(lib, gdn.dims(16, 32, 80)) == 3  # head_dim 80 unsupported
    assert _decode(lib, gdn.dims(16, 32, 128, map=7)) == 1
    assert _decode(lib, gdn.dims(16, 32, 128, decay=5)) == 1
    assert _decode(lib, gdn.dims(1, 32, 128)) == 3  # 32 V heads per K head > 16
    assert _decode(lib, ok, batch=-1) == 1
    assert _decode(lib, ok, batch=70000) == 2  # grid y limit
    assert _decode(lib, ok, batch=0) == 0  # nothing to do, nothing launched
    assert _decode(lib, ok, ptrs={"x": None}) == 1
    assert _decode(lib, ok, core=False) == 1  # neither core_out nor z
    assert _decode(lib, ok, ptrs={"a": 0x20008}) == 5  # misaligned
    # the state overlapping the conv state
    assert _decode(lib, ok, ptrs={"st": 0x1000000 + 64}) == 4
    # the core output overlapping an input
    assert _decode(lib, ok, ptrs={"core": 0x10000}) == 4


def _decode_slots(lib, d, batch=2, num_slots=4, ptrs=None):
    p = dict(sl=0x80000, x=0x10000, a=0x20000, b=0x30000, dp=0x40000, dt=0x50000, w=0x60000,
             cs=0x1000000, st=0x10000000, core=0x70000000, z=None, nw=None, out=None)
    if ptrs:
        p.update(ptrs)
    v = [VP(p[k]) if p[k] is not None else None for k in
         ("x", "a", "b", "dp", "dt", "w", "cs", "st", "core", "z", "nw", "out")]
    return lib.gdn_decode_step_slots(ctypes.byref(d), batch,
                                     VP(p["sl"]) if p["sl"] is not None else None, num_slots,
                                     *v, None)


@no_device
def test_decode_slots_rejects_bad_arguments(lib):
    ok = gdn.dims(16, 32, 128)
    assert _decode_slots(lib, ok, ptrs={"sl": None}) == 1  # no slot table
    assert _decode_slots(lib, ok, num_slots=-1) == 1
    assert _decode_slots(lib, ok, ptrs={"sl": 0x80004}) == 5  # misaligned table
    assert _decode_slots(lib, ok, batch=0) == 0  # nothing to do, nothing launched
    # the pool's size, not the batch, decides the state's extent: 4 slots of
    # 2 MiB reach past a conv state placed 4 MiB after the state's start
    assert _decode_slots(lib, ok, ptrs={"cs": 0x10000000 + (4 << 20)}) == 4
    # the slot table is an input: the core output must not overlap it
    assert _decode_slots(lib, ok, ptrs={"core": 0x80000}) == 4


@no_device
def test_decode_multi_rejects_bad_arguments(lib):
    ok = gdn.dims(16, 32, 128)

    def call(batch=2, tokens=4, **ptrs):
        p = dict(x=0x10000, a=0x2000000, b=0x3000000, dp=0x100000, dt=0x110000, w=0x120000,
                 cs=0x4000000, st=0x10000000, core=0x70000000)
        p.update(ptrs)
        return lib.gdn_decode_multi(ctypes.byref(ok), batch, tokens,
                                    *[VP(p[k]) if p[k] is not None else None for k in
                                      ("x", "a", "b", "dp", "dt", "w", "cs", "st", "core")],
                                    None, None, None, None)
    assert call(tokens=0) == 1
    assert call(tokens=9) == 3  # more than 8 tokens per call
    assert call(batch=0) == 0  # nothing to do, nothing launched
    assert call(x=None) == 1
    # the activations span B*T rows: 2 x 4 x 8192 bf16 = 128 KiB from 0x10000,
    # so a core output at 0x28000 overlaps them (with one token it would not)
    assert call(core=0x28000) == 4
    # more than 8 V heads per K head: one token runs, several do not
    wide = gdn.dims(1, 16, 128)
    args = [VP(a) for a in (0x10000, 0x2000000, 0x3000000, 0x100000, 0x110000, 0x120000, 0x4000000,
                            0x10000000, 0x70000000)] + [None] * 4
    assert lib.gdn_decode_multi(ctypes.byref(wide), 2, 2, *args) == 3
    args[8] = VP(0x10000)  # (the core output on the activations: refused on the host)
    assert lib.gdn_decode_multi(ctypes.byref(wide), 2, 1, *args) == 4


@no_device
def test_conv_and_prefill_and_norm_reject_bad_arguments(lib):
    d = gdn.dims(2, 4, 32)
    f = lib.gdn_conv_update
    assert f(ctypes.byref(d), -1, VP(0x100), 0, None, None, None, None, None) == 1
    assert f(ctypes.byref(d), 0, None, 5, None, None, None, None, None) == 1  # tokens, no seqs
    assert f(ctypes.byref(d), 0, None, 0, None, None, None, None, None) == 0
    assert f(ctypes.byref(d), 1, VP(0x100), 4, VP(0x1000), VP(0x9000), VP(0xa000),
             VP(0x1000 + 16), None) == 4  # y overlaps x
    assert f(ctypes.byref(d), 1, VP(0x104), 4, VP(0x1000), VP(0x9000), VP(0xa000),
             VP(0x100000), None) == 5  # cu_seqlens misaligned
    assert f(ctypes.byref(d), 1, VP(0x100), 2 ** 62, VP(0x1000), VP(0x9000), VP(0xa000),
             VP(0x100000), None) == 2  # extent overflow
    # the tiles' TMA row coordinates are int32: 2^31 - 65 tokens is the most
    big = 1 << 44
    assert f(ctypes.byref(d), 1, VP(0x100), 2 ** 31 - 64, VP(0x1000), VP(big), VP(big + 0x1000),
             VP(2 * big), None) == 2

    pf = lib.gdn_prefill_chunked
    base = [ctypes.byref(d), 1, VP(0x100), 10, VP(0x1000), 128, VP(0x2000), 128, VP(0x3000), 128,
            VP(0x4000), VP(0x5000), VP(0x6000), VP(0x7000), 0, VP(0x100000), VP(0x200000), None,
            None, None, None, 0, None]
    args = list(base)
    args[5] = 8  # q stride below Hk*D
    assert pf(*args) == 1
    args = list(base)
    args[5] = 68  # q stride not a multiple of 16 bytes
    assert pf(*args) == 5
    args = list(base)
    args[14] = 32  # unknown flag
    assert pf(*args) == 1
    args = list(base)
    args[14] = gdn.GDN_PREFILL_CARRY_WHOLE | gdn.GDN_PREFILL_CARRY_SLICED  # both carry kernels
    assert pf(*args) == 1
    args = list(base)
    args[16] = VP(0x100000)  # core_out aliases the state
    assert pf(*args) == 4
    args = list(base)
    args[15] = VP(0x1000)  # state overlaps q
    assert pf(*args) == 4

    # workspace: too small, misaligned, overlapping an input (bf16, D=128)
    d2 = gdn.dims(2, 4, 128, io_dtype=torch.bfloat16)
    need = ctypes.c_int64(0)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(d2), 1, 10, 0, ctypes.byref(need)) == 0
    assert need.value > 0
    wbase = [ctypes.byref(d2), 1, VP(0x100), 10, VP(0x10000), 256, VP(0x20000), 256,
             VP(0x30000), 512, VP(0x40000), VP(0x50000), VP(0x60000), VP(0x70000), 0,
             VP(0x1000000), VP(0x2000000), None, None, None]
    assert pf(*wbase, VP(0x4000000), need.value - 1, None) == 1  # too small
    assert pf(*wbase, VP(0x4000010), need.value, None) == 5  # not 256-byte aligned
    assert pf(*wbase, VP(0x30000), need.value, None) == 4  # overlaps v

    rn = lib.gdn_gated_rmsnorm
    assert rn(ctypes.byref(d), -1, None, None, None, None, None) == 1
    assert rn(ctypes.byref(d), 0, None, None, None, None, None) == 0
    assert rn(ctypes.byref(d), 4, VP(0x1000), VP(0x2000), VP(0x3000), VP(0x1000), None) == 4
    assert rn(ctypes.byref(d), 4, VP(0x1004), VP(0x2000), VP(0x3000), VP(0x9000), None) == 5


def test_binding_fails_loudly_on_cpu_tensors(lib):
    d = gdn.dims(2, 4, 32, io_dtype=torch.float32)
    t = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        gdn.gdn_gated_rmsnorm(d, t, t, torch.zeros(32), t)


def test_binding_checks_every_tensor_size_before_the_call(lib):
    """The C ABI sees only pointers: an undersized tensor must be caught in
    the binding (a kernel would otherwise read or write past it). Correctly
    sized CPU tensors get past these checks and fail on the device check."""
    f32 = torch.float32
    d = gdn.dims(2, 4, 32, io_dtype=f32)  # C = (2*2 + 4) * 32 = 256
    Z = torch.zeros

    def dec(**over):
        t = dict(x=Z(2, 256), a=Z(2, 4), b=Z(2, 4), dp=Z(4), dt=Z(4), w=Z(256, 4),
                 cs=Z(2, 256, 3), st=Z(2, 4, 32, 32), core=Z(2, 4, 32))
        t.update(over)
        gdn.gdn_decode_step(d, t["x"], t["a"], t["b"], t["dp"], t["dt"], t["w"], t["cs"],
                            t["st"], core_out=t["core"])

    for name, small in (("a", Z(1, 4)), ("b", Z(2, 3)), ("dp", Z(3)), ("w", Z(255, 4)),
                        ("cs", Z(1, 256, 3)), ("st", Z(1, 4, 32, 32)), ("core", Z(2, 4, 31))):
        with pytest.raises(ValueError, match="elements"):
            dec(**{name: small})
    with pytest.raises(ValueError, match="CUDA"):
        dec()

    def multi(**over):
        t = dict(x=Z(2, 3, 256), a=Z(2, 3, 4), b=Z(2, 3, 4), st=Z(2, 4, 32, 32),
                 core=Z(2, 3, 4, 32))
        t.update(over)
        gdn.gdn_decode_multi(d, t["x"], t["a"], t["b"], Z(4), Z(4), Z(256, 4), Z(2, 256, 3),
                             t["st"], core_out=t["core"])

    for name, small in (("a", Z(2, 2, 4)), ("core", Z(2, 2, 4, 32)), ("st", Z(1, 4, 32, 32))):
        with pytest.raises(ValueError, match="elements"):
            multi(**{name: small})
    with pytest.raises(ValueError, match="CUDA"):
        multi()

    slots = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="elements"):  # z of 1 row for 2
        gdn.gdn_decode_step_slots(d, slots, Z(2, 256), Z(2, 4), Z(2, 4), Z(4), Z(4), Z(256, 4),
                                  Z(5, 256, 3), Z(5, 4, 32, 32), z=Z(1, 4, 32), norm_w=Z(32),
                                  out=Z(2, 4, 32))

    def pre(**over):
        T = 10
        t = dict(q=Z(T, 64), k=Z(T, 64), v=Z(T, 128), a=Z(T, 4), st=Z(2, 4, 32, 32),
                 core=Z(T, 4, 32))
        t.update(over)
        cu = torch.tensor([0, 4, T], dtype=torch.int32)
        gdn.gdn_prefill_chunked(d, cu, t["q"], t["k"], t["v"], t["a"], Z(T, 4), Z(4), Z(4),
                                t["st"], core_out=t["core"], workspace=None)

    for name, small in (("k", Z(9, 64)), ("v", Z(10, 96)), ("a", Z(9, 4)),
                        ("st", Z(1, 4, 32, 32)), ("core", Z(9, 4, 32))):
        with pytest.raises(ValueError, match="rows|elements"):
            pre(**{name: small})
    with pytest.raises(ValueError, match="CUDA"):
        pre()

    cu = torch.tensor([0, 3], dtype=torch.int32)
    with pytest.raises(ValueError, match="elements"):
        gdn.gdn_conv_update(d, cu, Z(3, 256), Z(256, 4), Z(1, 256, 3), Z(2, 256))
    with pytest.raises(ValueError, match="elements"):
        gdn.gdn_gated_rmsnorm(d, Z(4, 32), Z(3, 32), Z(32), Z(4, 32))


def test_binding_static_scratch_size_matches_the_header():
    """The binding's GDN_STATIC_SCRATCH_BYTES is the header's."""
    with open(os.path.join(ROOT, "include", "gdn.h")) as f:
        text = f.read()
    m = re.search(r"#define GDN_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", text)
    assert m is not None
    assert gdn.GDN_STATIC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_selftest_wait_timeout_rejects_bad_arguments(lib):
    """Checked on the host before any launch: the limit's range and the
    output pointer."""
    f = lib.gdn_selftest_wait_timeout
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_int64, VP, VP]
    assert f(999, VP(0x1000), None) == 1
    assert f(10_000_000_001, VP(0x1000), None) == 1
    assert f(1_000_000, None, None) == 1


def test_linear_needs_no_workspace_and_rejects_bad_arguments(lib):
    """gdn_linear: narrow outputs sum their K splits inside a thread-block
    cluster, so the workspace size is 0 and NULL is accepted; sizes, strides
    and alignment are checked before anything is launched."""
    for mnk in ((1, 64, 64), (64, 2048, 4096), (128, 12352, 2048)):
        assert gdn.gdn_linear_workspace_size(*mnk) == 0
    f = lib.gdn_linear
    ok = [64, 2048, 4096, VP(0x10000), 4096, VP(0x100000000), None, VP(0x200000000), 2048, None, 0, None]
    bad = list(ok)
    bad[0] = 0  # no rows
    assert f(*bad) == 1
    bad = list(ok)
    bad[0] = 129  # more rows than one MMA
    assert f(*bad) == 1
    bad = list(ok)
    bad[1] = 96  # N not a multiple of 64
    assert f(*bad) == 1
    bad = list(ok)
    bad[4] = 4092  # x rows closer than K
    assert f(*bad) == 1
    bad = list(ok)
    bad[3] = VP(0x10008)  # x not 16-byte aligned
    assert f(*bad) == 5
    bad = list(ok)
    bad[7] = VP(0x10000 + 64)  # y overlapping x
    assert f(*bad) == 4
    d = gdn.dims(16, 32, 128)
    # the decode layer's workspace: the activations between its three calls only
    C, vw, Hv = (2 * 16 + 32) * 128, 32 * 128, 32
    align = lambda n: (n + 255) // 256 * 256
    B = 64
    expect = (align(B * C * 2) + align(B * vw * 2) + 2 * align(B * Hv * 2) + align(B * vw * 2))
    assert gdn.gdn_decode_layer_workspace_size(d, 2048, B) == expect


def test_host_pointer_rejects_null_and_the_binding_rejects_pageable_memory(lib):
    """gdn_host_pointer checks its arguments before any CUDA call; the
    binding takes pinned host memory only where the call allows it, and never
    pageable memory."""
    import torch
    import gated_delta_net_causal_gb300 as gdn
    out = ctypes.c_void_p()
    assert lib.gdn_host_pointer(None, ctypes.byref(out)) == 1
    buf = ctypes.create_string_buffer(64)
    assert lib.gdn_host_pointer(ctypes.cast(buf, ctypes.c_void_p), None) == 1
    d = gdn.dims(2, 4, 128, io_dtype=torch.bfloat16)
    C = gdn.gdn_qkv_features(d)
    bf, f32 = torch.bfloat16, torch.float32
    args = (torch.zeros(2, C, dtype=bf), torch.zeros(2, 4, dtype=bf), torch.zeros(2, 4, dtype=bf),
            torch.zeros(4), torch.zeros(4), torch.zeros(C, 4, dtype=bf),
            torch.zeros(2, C, 3, dtype=bf), torch.zeros(2, 4, 128, 128, dtype=f32))
    with pytest.raises(ValueError, match="pinned host memory"):
        gdn.gdn_decode_step(d, *args, core_out=torch.zeros(2, 4, 128))
