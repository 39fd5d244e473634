"""GPU parity of gdn_decode_step_slots (through the C ABI): batch rows that
name state slots of a larger pool, padded rows, and out-of-range slots,
against the fp64 oracle run on the gathered states."""

import numpy as np
import pytest
import torch

import gdn_inputs as gi
from tests.gpu_helpers import (DECODE_OUT_ABS, DECODE_STATE_REL, F64, assert_abs, assert_gated,
                               assert_state_rel, cuda, decode_reference)

pytestmark = pytest.mark.gpu


class SlotRunner:
    def __init__(self, shape, w, pool_cs, pool_S):
        import gated_delta_net_causal_gb300 as gdn
        self.gdn = gdn
        self.shape = shape
        self.d = gdn.dims(shape.n_k_heads, shape.n_v_heads, shape.head_dim, shape.map,
                          shape.decay, gi.DTYPES[shape.dtype])
        self.w = {k: cuda(getattr(w, k)) for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
        self.conv_state = cuda(pool_cs)
        self.state = cuda(pool_S)

    def step(self, x, slots):
        B, Hv, D = x.mixed_qkv.shape[0], self.shape.n_v_heads, self.shape.head_dim
        io = gi.DTYPES[self.shape.dtype]
        core_out = torch.full((B, Hv, D), float("nan"), device="cuda")
        out = torch.full((B, Hv, D), float("nan"), device="cuda", dtype=io)
        self.gdn.gdn_decode_step_slots(
            self.d, torch.as_tensor(slots, dtype=torch.int32).cuda(), cuda(x.mixed_qkv),
            cuda(x.a), cuda(x.b), self.w["decay_param"], self.w["dt_bias"], self.w["conv_w"],
            self.conv_state, self.state, core_out=core_out, z=cuda(x.z).view(B, Hv, D),
            norm_w=self.w["norm_w"], out=out)
        return core_out, out


def _run_pool(shape, pool, batch, tables, seed, check_rows=None):
    """Decode steps whose batch rows work on the slots `tables[step]` names.
    The oracle runs on its own pool's states of those slots; slots no row
    names must come out bit for bit as the previous step left them. With
    `check_rows`, only those rows are checked against the oracle, and the
    oracle's pool takes the GPU's states for the other live rows."""
    g = gi.rng(seed)
    w = gi.layer_weights(g, shape)
    cs0 = gi.conv_state(g, shape, pool, std=0.1)
    S0 = gi.delta_state(g, shape, pool, std=0.05)
    run = SlotRunner(shape, w, cs0, S0)
    cs, S = F64(cs0), F64(S0)          # the oracle's pool
    gS_prev, gcs_prev = S.copy(), cs.copy()  # the GPU's pool before the step
    for step, slots in enumerate(tables):
        assert len(slots) == batch
        x = gi.step_inputs(g, shape, batch)
        core_out, out = run.step(x, slots)
        torch.cuda.synchronize()
        live = [b for b in range(batch) if 0 <= slots[b] < pool]
        rows = live if check_rows is None else [b for b in live if b in check_rows]
        sl = [slots[b] for b in rows]
        rc, ry, ncs, nS = decode_reference(shape, w, x, cs[sl], S[sl], seqs=rows)
        tag = f"{shape} step {step}"
        co, oy = F64(core_out.cpu()), F64(out.cpu())
        assert_abs(co[rows], rc, DECODE_OUT_ABS, tag + " core")
        zr = F64(x.z).reshape(batch, shape.n_v_heads, shape.head_dim)[rows]
        assert_gated(oy[rows], ry, rc, zr, w.norm_w, shape.dtype, tag + " gated norm",
                     core_gpu=co[rows])
        pad = [b for b in range(batch) if b not in live]
        assert np.all(co[pad] == 0.0), tag + " padded core rows are zero"
        assert np.all(oy[pad] == 0.0), tag + " padded gated rows are zero"
        gS, gcs = F64(run.state.cpu()), F64(run.conv_state.cpu())
        named = {slots[b] for b in live}
        untouched = [s for s in range(pool) if s not in named]
        assert np.array_equal(gS[untouched], gS_prev[untouched]), tag + " untouched slots (state)"
        assert np.array_equal(gcs[untouched], gcs_prev[untouched]), tag + " untouched slots (conv)"
        assert_state_rel(gS[sl], nS, DECODE_STATE_REL, tag + " state")
        assert np.array_equal(gcs[sl], ncs), tag + " conv state (bitwise)"
        S[sl], cs[sl] = nS, ncs
        other = [slots[b] for b in live if b not in rows]
        S[other], cs[other] = gS[other], gcs[other]
        gS_prev, gcs_prev = gS, gcs
    assert run.gdn.gdn_device_error() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("mp,dec", [(gi.GROUPED, gi.LOG_RATE), (gi.TILED, gi.NEGATIVE_RATE)])
def test_slots_small_pool(dtype, mp, dec):
    shape = gi.Shape(4, 8, 128, map=mp, decay=dec, dtype=dtype)
    tables = [[7, -1, 2, 10, 0, 5],
              [10, 7, -3, 2, 8, -1],
              [1, 2, 3, 4, 5, 6]]
    _run_pool(shape, pool=11, batch=6, tables=tables, seed=4100 + mp * 10 + dec)


def test_slots_rep_eight_and_small_heads():
    _run_pool(gi.Shape(1, 8, 128, dtype="bf16"), pool=5, batch=3,
              tables=[[4, -1, 0], [0, 4, 2]], seed=4200)
    _run_pool(gi.Shape(2, 4, 64, dtype="f16"), pool=7, batch=4,
              tables=[[6, 1, -1, 3], [-1, -1, 6, 0]], seed=4201)


def test_slots_identity_table_matches_the_plain_call_bitwise():
    """slots = 0..B-1 over a pool of B is gdn_decode_step itself."""
    import gated_delta_net_causal_gb300 as gdn
    shape = gi.Shape(4, 8, 128, map=gi.TILED, decay=gi.NEGATIVE_RATE, dtype="bf16")
    B = 5
    g = gi.rng(4300)
    w = gi.layer_weights(g, shape)
    cs0 = cuda(gi.conv_state(g, shape, B, std=0.1))
    S0 = cuda(gi.delta_state(g, shape, B, std=0.05))
    x = gi.step_inputs(g, shape, B)
    d = gdn.dims(4, 8, 128, gi.TILED, gi.NEGATIVE_RATE, torch.bfloat16)
    wd = {k: cuda(getattr(w, k)) for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
    res = []
    for use_slots in (False, True):
        cs, S = cs0.clone(), S0.clone()
        core = torch.empty((B, 8, 128), device="cuda")
        out = torch.empty((B, 8, 128), device="cuda", dtype=torch.bfloat16)
        args = (cuda(x.mixed_qkv), cuda(x.a), cuda(x.b), wd["decay_param"], wd["dt_bias"],
                wd["conv_w"], cs, S)
        kw = dict(core_out=core, z=cuda(x.z).view(B, 8, 128), norm_w=wd["norm_w"], out=out)
        if use_slots:
            gdn.gdn_decode_step_slots(d, torch.arange(B, dtype=torch.int32, device="cuda"),
                                      *args, **kw)
        else:
            gdn.gdn_decode_step(d, *args, **kw)
        torch.cuda.synchronize()
        res.append((core, out, cs, S))
    for a, b in zip(*res):
        assert torch.equal(a, b)


def test_slot_out_of_range_is_skipped_and_recorded():
    """An entry >= num_slots is caught by the kernel's own bounds check: the
    row is skipped like a padded one and GDN_ERR_EXTENT is recorded."""
    import gated_delta_net_causal_gb300 as gdn
    shape = gi.Shape(2, 4, 128, dtype="bf16")
    g = gi.rng(4400)
    w = gi.layer_weights(g, shape)
    run = SlotRunner(shape, w, gi.conv_state(g, shape, 3, std=0.1),
                     gi.delta_state(g, shape, 3, std=0.05))
    assert gdn.gdn_device_error(clear=True) == 0
    before_S, before_cs = run.state.clone(), run.conv_state.clone()
    x = gi.step_inputs(g, shape, 2)
    core_out, out = run.step(x, [1, 3])
    torch.cuda.synchronize()
    assert gdn.gdn_device_error(clear=True) == 2  # GDN_ERR_EXTENT
    assert gdn.gdn_device_error() == 0
    assert torch.equal(run.state[0], before_S[0]) and torch.equal(run.state[2], before_S[2])
    assert torch.equal(run.conv_state[0], before_cs[0])
    assert not torch.equal(run.state[1], before_S[1])
    assert torch.all(core_out[1] == 0) and torch.all(out[1] == 0)


def test_slots_full_size_batch_in_a_pool():
    """The batched-decode shape (B=64, Hk=16, Hv=32, D=128, Tiled,
    negative-rate, bf16) scattered over a pool of 256 slots with every fourth
    row padded; the oracle checks sampled rows, the rest must leave every
    slot no row names untouched."""
    shape = gi.Shape(16, 32, 128, map=gi.TILED, decay=gi.NEGATIVE_RATE, dtype="bf16")
    rs = np.random.default_rng(4500)
    tables = []
    for _ in range(2):
        perm = rs.permutation(256)[:64].tolist()
        tables.append([-1 if b % 4 == 3 else perm[b] for b in range(64)])
    _run_pool(shape, pool=256, batch=64, tables=tables, seed=4501, check_rows={0, 17, 42, 62})
