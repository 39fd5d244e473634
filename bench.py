"""Benchmark of the GB300 gated delta-net core.

Headline workload (one step = one fused gdn_decode_step over the batch: conv +
SiLU, split, q/k l2 norm, gates, the delta-rule update of the fp32 state in
place, and the gated RMSNorm epilogue):
  batched decode, B=64 sequences x 1 token, Hk=16, Hv=32, D=128, Tiled map,
  negative-rate decay, bf16 activations ~N(0,1), fp32 state ~N(0,0.02)
  (128 MiB), conv state bf16 ~N(0,0.1); 16 distinct input sets cycled.
Metric: state GB/s = 2 * B * Hv * D^2 * 4 bytes / step time.

A second block measures chunked prefill (one sequence of T=4096, Hk=16, Hv=32,
D=128, Grouped, bf16 raw q/k/v/z/a/b, fused gated RMSNorm) in tokens/s, with
its tensor roofline, the same call end to end from host buffers, and the
oracle's rate on the host cores; a third the whole path on the varlen workload
(conv update over 8 packed sequences, chunked prefill with the fused norm, 16
decode steps) in tokens/s, with the prefill call alone against its roofline;
a fourth the batch-1 layer's latency (four decode steps, one multi-token call,
the 3 + 1 split through conv update and chunked prefill).

Timing: W untimed warm-up steps, then K steps each bracketed by CUDA events on
the launching stream; a 512 MiB buffer is overwritten between timed steps so
no step starts with the previous step's state in L2. Under torchrun each rank
runs its own batch (weak scaling, no collective on the data path); the step
time is the max over ranks.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload instead (the CPU baseline).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gdn_inputs as gi  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")
DECODE_WORKLOAD = ("batched decode B=64 x 1 token, Hk=16 Hv=32 D=128, Tiled, negative-rate, "
                   "bf16 activations, fp32 state")
PREFILL_WORKLOAD = "chunked prefill N=1 T=4096, Hk=16 Hv=32 D=128, Grouped, log-rate, bf16"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def _kernel_hash(*files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "gated_delta_net_causal_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _profile_traffic(name: str, khash: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    path = os.path.join(PROFILES, name)
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                kv[k.strip()] = v.strip()
    if kv.get("kernel_hash") != khash:
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier_max(value: float, ws: int) -> float:
    """The maximum of `value` over all ranks (the slowest rank's time), after
    a barrier; the value itself with one process."""
    if ws == 1:
        return value
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], device=dev, dtype=torch.float64)
    dist.barrier()
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------- GPU arm

def _decode_setup(batch: int, sets: int, rank: int):
    """Rank r runs its own `batch` sequences (global sequences r*batch ..
    (r+1)*batch - 1, drawn from the rank's own seed): the sequences are
    sharded across ranks with no exchange."""
    import gated_delta_net_causal_gb300 as gdn
    wl = gi.workload_batched_decode(batch=batch, sets=sets, shard=rank)
    shape, w = wl["shape"], wl["weights"]
    d = gdn.dims(16, 32, 128, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    dev = {k: getattr(w, k).cuda() for k in ("conv_w", "decay_param", "dt_bias", "norm_w")}
    steps = [{"x": s.mixed_qkv.cuda(), "a": s.a.cuda(), "b": s.b.cuda(),
              "z": s.z.cuda().view(batch, 32, 128)} for s in wl["steps"]]
    host = [{"x": s.mixed_qkv.pin_memory(), "a": s.a.pin_memory(), "b": s.b.pin_memory(),
             "z": s.z.pin_memory()} for s in wl["steps"]]
    state = wl["state"].cuda()
    cstate = wl["conv_state"].cuda()
    out = torch.empty((batch, 32, 128), device="cuda", dtype=torch.bfloat16)
    return gdn, d, dev, steps, host, state, cstate, out, shape


def _decode_call(gdn, d, dev, inp, state, cstate, out):
    gdn.gdn_decode_step(d, inp["x"], inp["a"], inp["b"], dev["decay_param"], dev["dt_bias"],
                        dev["conv_w"], cstate, state, core_out=None, z=inp["z"],
                        norm_w=dev["norm_w"], out=out)


def run_gpu(args, ws, rank, local):
    torch.cuda.set_device(local)
    peaks = _peaks()
    only = "prefill" if args.prefill_only else args.only
    if only:
        blocks = {"prefill": lambda: run_prefill(args, peaks, ws),
                  "varlen_path": lambda: run_varlen(args, ws, peaks),
                  "decode_layer": lambda: run_decode_layer(args, ws, peaks),
                  "multi_token_decode": lambda: run_multi_decode(args, ws, peaks),
                  "slot_decode": lambda: run_slot_decode(args, ws, peaks)}
        line = {"metric": f"the {only} block alone", only: blocks[only]()}
        return line if rank == 0 else None
    batch = args.batch
    gdn, d, dev, steps, host, state, cstate, out, shape = _decode_setup(batch, 16, rank)
    flush = torch.empty(512 * 1024 * 1024 // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    B, Hv, D, C = batch, 32, 128, shape.qkv_features
    state_bytes = 2 * B * Hv * D * D * 4
    other_bytes = (B * C * 2 + 2 * B * Hv * 2 + B * Hv * D * 2 + 2 * B * C * 3 * 2
                   + B * Hv * D * 2 + C * 4 * 2 + 3 * Hv * 4 + D * 4)

    # Each step works on one of `nsets` state (and conv-state) sets in turn,
    # nsets x 128 MiB >= 512 MiB: a step's state was last touched nsets steps
    # earlier and the traffic since has evicted it from L2, as between two
    # steps of one layer in a model. Activations cycle through 16 step sets.
    nsets = max(4, -(-512 * 2**20 // state.nbytes))
    states = [state] + [state.clone() for _ in range(nsets - 1)]
    cstates = [cstate] + [cstate.clone() for _ in range(nsets - 1)]

    def dstep(i):
        _decode_call(gdn, d, dev, steps[i % 16], states[i % nsets], cstates[i % nsets], out)

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(args.warmup):
        dstep(i)
    torch.cuda.synchronize()

    # The K timed steps run back to back, as a serving loop issues them: one
    # CUDA graph holding the K consecutive gdn_decode_step calls, captured
    # and replayed once (untimed) before the timed replay.
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(args.steps):
                dstep(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    flush.fill_(0.0)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    t_step = _barrier_max(ev0.elapsed_time(ev1) * 1e-3 / args.steps, ws)
    ms_per_step = t_step * 1e3
    del graph

    # The same steps timed one launch at a time, a 512 MiB buffer overwritten
    # before each: every launch pays its own start-up and drain (~5.6 us
    # here, the same for a plain copy of the same bytes).
    n_iso = min(args.steps, 64)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_iso)]
    for i in range(n_iso):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        dstep(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_iso = _barrier_max(statistics.mean(a.elapsed_time(b) * 1e-3 for a, b in ev), ws)

    # Yardstick: a plain device copy of the state's bytes (read + write =
    # state_bytes), timed both ways.
    src = [torch.empty(state.numel(), device="cuda") for _ in range(nsets)]
    dst = [torch.empty(state.numel(), device="cuda") for _ in range(nsets)]
    for t in src:
        t.fill_(1.0)

    def cstep(i):
        dst[i % nsets].copy_(src[i % nsets])

    for i in range(nsets):
        cstep(i)
    side.wait_stream(stream)
    cgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(cgraph, stream=side):
            for i in range(args.steps):
                cstep(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    cgraph.replay()
    flush.fill_(0.0)
    ev0.record(stream)
    cgraph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t_copy = _barrier_max(ev0.elapsed_time(ev1) * 1e-3 / args.steps, ws)
    for i in range(n_iso):
        flush.fill_(float(i))
        ev[i][0].record(stream)
        cstep(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    t_copy_iso = _barrier_max(statistics.mean(a.elapsed_time(b) * 1e-3 for a, b in ev), ws)
    del cgraph, src, dst, states[1:], cstates[1:]
    torch.cuda.empty_cache()

    # end to end through the C ABI with host buffers: H2D of the step's
    # activations from pinned memory, the call, D2H of the gated output, then
    # a host sync, every step. As a serving loop would issue it: one CUDA
    # graph per input set holding the copies and the call (captured once,
    # outside the timed region), replayed per step; the same sequence issued
    # eagerly, call by call, is reported beside it.
    out_host = torch.empty((B, Hv, D), dtype=torch.bfloat16).pin_memory()
    e2e_steps = min(args.steps, 64)
    # a step's activations packed into one pinned buffer (x | a | b | z, each
    # part 16-byte aligned) and moved by one copy into one device buffer the
    # call reads views of
    names = ("x", "a", "b", "z")
    offs, total = {}, 0
    for k in names:
        offs[k] = total
        total += (host[0][k].numel() * host[0][k].element_size() + 15) // 16 * 16
    packed = []
    for i in range(16):
        hp = torch.empty(total, dtype=torch.uint8).pin_memory()
        for k in names:
            nb = host[i][k].numel() * host[i][k].element_size()
            hp[offs[k]:offs[k] + nb].copy_(host[i][k].reshape(-1).view(torch.uint8))
        packed.append(hp)
    dpack = torch.empty(total, dtype=torch.uint8, device="cuda")

    def dview(k):
        t = host[0][k]
        nb = t.numel() * t.element_size()
        return dpack[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)

    dbuf = {k: dview(k) for k in names}
    h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in names)
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step(i):
        dpack.copy_(packed[i % 16], non_blocking=True)
        _decode_call(gdn, d, dev, {"x": dbuf["x"], "a": dbuf["a"], "b": dbuf["b"],
                                   "z": dbuf["z"].view(B, Hv, D)}, state, cstate, out)
        out_host.copy_(out, non_blocking=True)

    torch.cuda.synchronize()
    eager_times = []
    for i in range(e2e_steps):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        e2e_step(i)
        torch.cuda.synchronize()
        eager_times.append(time.perf_counter() - t0)
    graphs = []
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for i in range(16):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                e2e_step(i)
            graphs.append(g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    e2e_times = []
    for i in range(e2e_steps):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        graphs[i % 16].replay()
        torch.cuda.synchronize()
        e2e_times.append(time.perf_counter() - t0)
    t_e2e = _barrier_max(statistics.mean(e2e_times), ws)
    t_eager = _barrier_max(statistics.mean(eager_times), ws)

    # the same steps with no copies: the call reads the step's x, a, b, z
    # from the packed pinned buffer and writes the gated output into pinned
    # host memory itself, over the host link (gdn_decode_step takes mapped
    # pinned host memory for its activations and outputs); one CUDA graph per
    # input set holding only the call, replayed per step, host sync per step
    def hview(hp, k):
        t = host[0][k]
        nb = t.numel() * t.element_size()
        return hp[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)

    def mapped_step(i):
        hp = packed[i % 16]
        _decode_call(gdn, d, dev, {"x": hview(hp, "x"), "a": hview(hp, "a"), "b": hview(hp, "b"),
                                   "z": hview(hp, "z").view(B, Hv, D)}, state, cstate, out_host)

    mgraphs = []
    with torch.cuda.stream(side):
        for i in range(16):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                mapped_step(i)
            mgraphs.append(g)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    mapped_times = []
    for i in range(e2e_steps):
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        mgraphs[i % 16].replay()
        torch.cuda.synchronize()
        mapped_times.append(time.perf_counter() - t0)
    t_mapped = _barrier_max(statistics.mean(mapped_times), ws)
    del graphs, mgraphs

    # chunked prefill block and the varlen whole-path block
    prefill = run_prefill(args, peaks, ws) if not args.no_prefill else None
    varlen = run_varlen(args, ws, peaks) if not args.no_prefill else None
    batch1 = run_batch1(args, ws) if not args.no_prefill else None
    layer = run_decode_layer(args, ws, peaks) if not args.no_extra else None
    multilayer = run_multilayer(args, ws, peaks) if not args.no_multilayer else None
    slot_dec = run_slot_decode(args, ws, peaks) if not args.no_extra else None
    multi_dec = run_multi_decode(args, ws, peaks) if not args.no_extra else None
    clk = clocks.stop()
    if clk is not None:
        clk["window"] = "decode warm-up through the prefill blocks (brackets the timed steps)"

    if rank != 0:
        return None
    value = ws * state_bytes / t_step / 1e9
    achieved = (state_bytes + other_bytes) / t_step / 1e9
    khash = _kernel_hash("decode.cu", "gdn_common.cuh")
    line = {
        "metric": "GDN decode state GB/s (% HBM peak); chunked prefill tokens/s (% roofline)",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": DECODE_WORKLOAD, "batch_per_gpu": B, "global_batch": B * ws,
                   "n_k_heads": 16, "n_v_heads": 32, "head_dim": 128,
                   "state_bytes_per_step": state_bytes,
                   "l2": f"inputs larger than L2: {nsets} state and conv-state sets of "
                         f"{state.nbytes >> 20} MiB cycled step by step (each step's state last "
                         f"touched {nsets} steps earlier); 512 MiB overwritten before the timed "
                         "region",
                   "timing": f"the {args.steps} consecutive steps as one CUDA graph replay between "
                             "two CUDA events; ms_per_step = that time / steps",
                   "parallelism": f"replicas x{ws} (sequences sharded, no collective)"},
        "seq_per_s": round(ws * B / t_step, 1),
        "hbm_frac_state": round(value / ws / peaks["hbm_gbs"], 4),
        "isolated_step": {"value": round(ws * state_bytes / t_iso / 1e9, 2), "unit": "GB/s",
                          "ms_per_step": round(t_iso * 1e3, 5),
                          "hbm_frac_state": round(state_bytes / t_iso / 1e9 / peaks["hbm_gbs"], 4),
                          "timing": f"{n_iso} launches, each between two CUDA events with a "
                                    "512 MiB buffer overwritten before it"},
        "same_bytes_copy": {"bytes": state_bytes,
                            "back_to_back_us": round(t_copy * 1e6, 2),
                            "back_to_back_frac": round(state_bytes / t_copy / 1e9 / peaks["hbm_gbs"], 4),
                            "isolated_us": round(t_copy_iso * 1e6, 2),
                            "isolated_frac": round(state_bytes / t_copy_iso / 1e9 / peaks["hbm_gbs"], 4),
                            "what": "torch device copy of the state's size, timed both ways "
                                    "(yardstick, not part of the step)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "traffic": _profile_traffic("decode_step_b64.txt", khash),
                     "peak_source": peaks["source"], "kernel": "decode_step_kernel<bf16,128>",
                     "algorithmic_bytes_per_launch": state_bytes + other_bytes},
        "e2e": {"value": round(ws * state_bytes / t_e2e / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(t_e2e * 1e3, 4),
                "issue": "one CUDA graph per input set (one H2D copy of the step's x, a, b, z packed "
                         "in one pinned buffer, the gdn_decode_step call on views of the device "
                         "buffer, D2H of the gated output), replayed per step, host sync per step",
                "eager": {"value": round(ws * state_bytes / t_eager / 1e9, 2), "unit": "GB/s",
                          "ms_per_step": round(t_eager * 1e3, 4)},
                "host_mapped": {"value": round(ws * state_bytes / t_mapped / 1e9, 2),
                                "unit": "GB/s", "ms_per_step": round(t_mapped * 1e3, 4),
                                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                                "issue": "no copies: the gdn_decode_step call reads x, a, b, z "
                                         "from the packed pinned host buffer and writes the gated "
                                         "output to pinned host memory over the host link; one "
                                         "CUDA graph per input set holding only the call, host "
                                         "sync per step"}},
        "gpu_launches": args.steps,
        "clocks": clk,
    }
    if prefill is not None:
        line["prefill"] = prefill
    if varlen is not None:
        line["varlen_path"] = varlen
    if batch1 is not None:
        line["batch1_layer"] = batch1
    if layer is not None:
        line["decode_layer"] = layer
    if multilayer is not None:
        line["multilayer_decode"] = multilayer
    if slot_dec is not None:
        line["slot_decode"] = slot_dec
    if multi_dec is not None:
        line["multi_token_decode"] = multi_dec
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline_decode(seconds=args.cpu_seconds)
    return line


def run_prefill(args, peaks, ws):
    import gated_delta_net_causal_gb300 as gdn
    T = 4096
    wl = gi.workload_prefill(T, random_state=True)
    shape, w = wl["shape"], wl["weights"]
    d = gdn.dims(16, 32, 128, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    q, k, v = (wl[n].cuda().view(T, -1) for n in ("q", "k", "v"))
    a, b, z = wl["a"].cuda(), wl["b"].cuda(), wl["z"].cuda()
    dp, dt, nw = w.decay_param.cuda(), w.dt_bias.cuda(), w.norm_w.cuda()
    cu = wl["cu_seqlens"].cuda()
    s0 = wl["state"].cuda()
    state = s0.clone()
    out = torch.empty((T, 32, 128), device="cuda", dtype=torch.bfloat16)
    wsb = torch.empty(gdn.gdn_prefill_workspace_size(d, 1, T), device="cuda", dtype=torch.uint8)
    flush = torch.empty(512 * 1024 * 1024 // 4, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()

    def call(flags=0):
        gdn.gdn_prefill_chunked(d, cu, q, k, v, a, b, dp, dt, state, core_out=None, z=z,
                                norm_w=nw, out=out, workspace=wsb, flags=flags)

    def timed(flags, n, graph):
        # graph: the call captured once as a CUDA graph (its tensor maps
        # encoded at capture) and each timed call one replay, so the host's
        # submission work is outside the events; else one eager call
        for _ in range(3):
            state.copy_(s0)
            call(flags)
        torch.cuda.synchronize()
        run = lambda: call(flags)
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                call(flags)
            torch.cuda.synchronize()
            run = g.replay
        times = []
        for i in range(n):
            state.copy_(s0)
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e-3)
        return _barrier_max(statistics.mean(times), ws)

    n = max(3, min(args.steps, 20))
    t = timed(0, n, True)
    t_eager = timed(0, n, False)
    # the library's default carry for one sequence of 32 V heads: the sliced
    # one (4 CTAs per V head) when Hv N <= 64 and 4 Hv N <= 2 x SMs, its
    # gated norm then a separate pass; the whole-row carry timed beside it
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    sliced = 32 * 1 <= 64 and 4 * 32 <= 2 * sms
    t_whole = timed(gdn.GDN_PREFILL_CARRY_WHOLE, n, True)

    # end to end through the C ABI with host buffers: the call's inputs (q, k,
    # v, a, b, z) packed in one pinned buffer and moved by one copy into one
    # device buffer the call reads views of, the call, the gated output copied
    # back, a host sync; the three captured once as a CUDA graph and replayed
    # per call (as the decode line's e2e); the state stays resident
    hsrc = {"q": wl["q"].view(T, -1), "k": wl["k"].view(T, -1), "v": wl["v"].view(T, -1),
            "a": wl["a"], "b": wl["b"], "z": wl["z"]}
    offs, total = {}, 0
    for nm, tt in hsrc.items():
        offs[nm] = total
        total += (tt.numel() * tt.element_size() + 255) // 256 * 256
    hpack = torch.empty(total, dtype=torch.uint8).pin_memory()
    for nm, tt in hsrc.items():
        nb = tt.numel() * tt.element_size()
        hpack[offs[nm]:offs[nm] + nb].copy_(tt.reshape(-1).view(torch.uint8))
    dpack = torch.empty(total, dtype=torch.uint8, device="cuda")
    dbuf = {nm: dpack[offs[nm]:offs[nm] + tt.numel() * tt.element_size()].view(tt.dtype).view(tt.shape)
            for nm, tt in hsrc.items()}
    out_host = torch.empty((T, 32, 128), dtype=torch.bfloat16).pin_memory()
    h2d = sum(tt.numel() * tt.element_size() for tt in hsrc.values())
    d2h = out_host.numel() * out_host.element_size()

    def e2e_call():
        dpack.copy_(hpack, non_blocking=True)
        gdn.gdn_prefill_chunked(d, cu, dbuf["q"], dbuf["k"], dbuf["v"], dbuf["a"], dbuf["b"], dp, dt,
                                state, core_out=None, z=dbuf["z"], norm_w=nw, out=out,
                                workspace=wsb)
        out_host.copy_(out, non_blocking=True)

    state.copy_(s0)
    e2e_call()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        ge = torch.cuda.CUDAGraph()
        with torch.cuda.graph(ge, stream=side):
            e2e_call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    e2e_times = []
    for i in range(max(3, min(args.steps, 10)) + 2):
        state.copy_(s0)
        flush.fill_(float(i))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ge.replay()
        torch.cuda.synchronize()
        e2e_times.append(time.perf_counter() - t0)
    t_e2e = _barrier_max(statistics.mean(e2e_times[2:]), ws)
    Hk, Hv, D, Cc = 16, 32, 128, 64
    flop_per_token = Hv * (6 * D * D + 6 * Cc * D + Cc * Cc / 3) + Hk * 4 * Cc * D
    flops = flop_per_token * T
    byts = T * (2 * Hk * D + 2 * Hv * D) * 2 + T * Hv * D * 2 + 2 * Hv * D * D * 4 + 4 * T * Hv * 2
    res = {"workload": PREFILL_WORKLOAD, "value": round(ws * T / t, 1), "unit": "tokens/s",
            "ms_per_call": round(t * 1e3, 4), "calls": n, "launches_per_call": 4 if sliced else 3,
            "carry": ("sliced: cp_slice_kernel, 4 CTAs per V head, then cp_norm_kernel" if sliced
                      else "whole rows: cp_chain_kernel, 1 CTA per V head"),
            "whole_row_carry_ms_per_call": round(t_whole * 1e3, 4),
            "eager_ms_per_call": round(t_eager * 1e3, 4),
            "timing": "one call per timed region (state reset, 512 MiB overwritten before it): the "
                      "call captured once as a CUDA graph and replayed between two CUDA events; "
                      "eager_ms_per_call times the same call issued from the host between the "
                      "events (host submission included)",
            "roofline": {"bound": "tensor", "achieved": round(flops / t / 1e12, 3),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(flops / t / 1e12 / peaks["bf16_tflops"], 5),
                         "traffic": _profile_traffic("prefill_cp_t4096.txt",
                                                     _kernel_hash("prefill_cp.cu", "tc_common.cuh",
                                                                  "gdn_common.cuh")),
                         "traffic_unit": "bytes per call (all launches)",
                         "peak_source": peaks["source"],
                         "algorithmic_flops_per_call": flops,
                         "algorithmic_bytes_per_call": byts,
                         "hbm_frac": round(byts / t / 1e9 / peaks["hbm_gbs"], 4),
                         "timed": "the whole call (chunk index, prep, carry, norm launches), "
                                  "graph replay",
                         "kernel": ("cp_prep_kernel + cp_slice_kernel + cp_norm_kernel" if sliced
                                    else "cp_prep_kernel + cp_chain_kernel")},
           "e2e": {"value": round(ws * T / t_e2e, 1), "unit": "tokens/s",
                   "ms_per_call": round(t_e2e * 1e3, 4), "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h,
                   "issue": "one H2D copy of q, k, v, a, b, z packed in one pinned buffer, the "
                            "gdn_prefill_chunked call on views of the device buffer, D2H of the "
                            "gated output, as one CUDA graph replayed per call; host sync per call"}}
    if not args.no_cpu_baseline and ws == 1:
        res["cpu_baseline"] = cpu_baseline_prefill(wl, seconds=min(args.cpu_seconds, 15.0))
    return res


def run_varlen(args, ws, peaks):
    """The whole hot path on the varlen workload: conv update over 8 packed
    sequences (lengths U[512,8192] as drawn, 34,482 tokens), chunked prefill
    with the fused gated norm continuing from their states, then 16 batched
    decode steps. Inputs are drawn on the device (same shapes and laws as the
    parity test's host-drawn ones)."""
    import gated_delta_net_causal_gb300 as gdn
    lengths = gi.varlen_lengths(gi.SEED_BASE + 5, 8, 512, 8192)
    N, T = len(lengths), int(sum(lengths))
    Hk, Hv, D = 16, 64, 128
    C = (2 * Hk + Hv) * D
    gen = torch.Generator(device="cuda").manual_seed(gi.SEED_BASE + 5)
    bf = torch.bfloat16

    def rn(*shape, std=1.0, dtype=bf):
        return (torch.randn(shape, device="cuda", generator=gen) * std).to(dtype)
    x, a, b, z = rn(T, C), rn(T, Hv), rn(T, Hv), rn(T, Hv, D)
    dec = [(rn(N, C), rn(N, Hv), rn(N, Hv), rn(N, Hv, D)) for _ in range(16)]
    conv_w = rn(C, 4, std=0.16)
    dp = torch.log(torch.rand(Hv, device="cuda", generator=gen) * 15 + 1)
    dt = torch.rand(Hv, device="cuda", generator=gen) - 0.5
    nw = (0.82 + 0.013 * torch.arange(D, device="cuda")).float()
    cs0, s0 = rn(N, C, 3, std=0.1), rn(N, Hv, D, D, std=0.02, dtype=torch.float32)
    cu = gi.cu_seqlens(lengths).cuda()
    d = gdn.dims(Hk, Hv, D, map=gdn.GDN_MAP_TILED, decay=gdn.GDN_DECAY_LOG_RATE, io_dtype=bf)
    y = torch.empty_like(x)
    out = torch.empty((T, Hv, D), device="cuda", dtype=bf)
    dout = torch.empty((N, Hv, D), device="cuda", dtype=bf)
    cs, st = cs0.clone(), s0.clone()
    qk = Hk * D
    wsb = torch.empty(gdn.gdn_prefill_workspace_size(d, N, T), device="cuda", dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def path():
        gdn.gdn_conv_update(d, cu, x, conv_w, cs, y)
        gdn.gdn_prefill_chunked(d, cu, y[:, :qk], y[:, qk:2 * qk], y[:, 2 * qk:], a, b, dp, dt,
                                st, z=z, norm_w=nw, out=out, workspace=wsb)
        for (xd, ad, bd, zd) in dec:
            gdn.gdn_decode_step(d, xd, ad, bd, dp, dt, conv_w, cs, st, z=zd, norm_w=nw, out=dout)

    def graphed(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g.replay

    def time_calls(run, reset, n):
        times = []
        for _ in range(n):
            reset()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1) * 1e-3)
        return times

    def reset_all():
        cs.copy_(cs0)
        st.copy_(s0)

    path()
    torch.cuda.synchronize()
    t_eager = _barrier_max(statistics.mean(time_calls(path, reset_all, 3)), ws)
    path_g = graphed(path)
    t = _barrier_max(statistics.mean(time_calls(path_g, reset_all, 3)), ws)
    tokens = T + 16 * N

    # the prefill call alone (the core of the path), on the conv output of the
    # first pass, the states reset before each call
    def pre():
        gdn.gdn_prefill_chunked(d, cu, y[:, :qk], y[:, qk:2 * qk], y[:, 2 * qk:], a, b, dp, dt,
                                st, z=z, norm_w=nw, out=out, workspace=wsb)

    pre_g = graphed(pre)
    tp = _barrier_max(statistics.mean(time_calls(pre_g, lambda: st.copy_(s0), 4)[1:]), ws)

    # the conv update alone (two launches: the outputs, then the state), the
    # conv states reset before each call
    conv_g = graphed(lambda: gdn.gdn_conv_update(d, cu, x, conv_w, cs, y))
    tc = _barrier_max(statistics.mean(time_calls(conv_g, lambda: cs.copy_(cs0), 4)[1:]), ws)
    cbytes = 2 * T * C * 2 + 2 * N * C * 3 * 2 + C * 4 * 2
    Cc = 64
    flops = T * (Hv * (6 * D * D + 6 * Cc * D + Cc * Cc / 3) + Hk * 4 * Cc * D)
    byts = (T * (2 * Hk * D + 2 * Hv * D) * 2 + T * Hv * D * 2 + 2 * N * Hv * D * D * 4
            + 2 * T * Hv * 2)
    return {"workload": "varlen: 8 sequences (34,482 tokens) conv update + chunked prefill with "
                        "fused norm + 16 decode steps, Hk=16 Hv=64 D=128, Tiled, bf16",
            "value": round(ws * tokens / t, 1), "unit": "tokens/s", "ms_per_pass": round(t * 1e3, 4),
            "eager_ms_per_pass": round(t_eager * 1e3, 4),
            "timing": "each pass, call or update captured once as a CUDA graph and replayed between "
                      "two CUDA events, states reset before each; eager_ms_per_pass issues the pass "
                      "from the host between the events",
            "launches_per_pass": 2 + 3 + 16,
            "prefill_core": {"value": round(ws * T / tp, 1), "unit": "tokens/s",
                             "ms_per_call": round(tp * 1e3, 4),
                             "roofline": {"bound": "tensor", "achieved": round(flops / tp / 1e12, 3),
                                          "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                          "frac": round(flops / tp / 1e12 / peaks["bf16_tflops"], 5),
                                          "algorithmic_flops_per_call": flops,
                                          "algorithmic_bytes_per_call": byts,
                                          "hbm_frac": round(byts / tp / 1e9 / peaks["hbm_gbs"], 4),
                                          "peak_source": peaks["source"]},
                             "timed": "the gdn_prefill_chunked call alone (index, prep, chain), "
                                      "fused norm, states reset before each of 3 timed replays"},
            "conv_update": {"us_per_call": round(tc * 1e6, 2),
                            "roofline": {"bound": "hbm", "achieved": round(cbytes / tc / 1e9, 1),
                                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                         "frac": round(cbytes / tc / 1e9 / peaks["hbm_gbs"], 4),
                                         "algorithmic_bytes_per_call": cbytes,
                                         "peak_source": peaks["source"]},
                            "kernel": "conv_fwd_kernel + conv_state_kernel",
                            "timed": "the gdn_conv_update call alone, conv states reset before "
                                     "each of 3 timed replays"}}


def run_batch1(args, ws):
    """The batch-1 layer (Hk=16, Hv=32, D=128, Grouped, log-rate, f16, the
    seeded inputs of the parity test): four tokens through gdn_decode_step one
    at a time, the same four as one gdn_decode_multi call, and the 3 + 1 split
    (conv update + chunked prefill on three tokens, then one decode step).
    Latency per pass, with the states reset before each pass; eager launches
    and, for the four steps, one CUDA graph."""
    import gated_delta_net_causal_gb300 as gdn
    wl = gi.workload_single_layer_b1(dtype="f16")
    shape, w, x = wl["shape"], wl["weights"], wl["inputs"]
    Hk, Hv, D = 16, 32, 128
    C = shape.qkv_features
    d = gdn.dims(Hk, Hv, D, map=shape.map, decay=shape.decay, io_dtype=torch.float16)
    xs, a, b = x.mixed_qkv.cuda(), x.a.cuda(), x.b.cuda()
    z = x.z.cuda().view(4, Hv, D)
    cw, dp, dt, nw = (getattr(w, n).cuda() for n in ("conv_w", "decay_param", "dt_bias", "norm_w"))
    cs0, s0 = wl["conv_state"].cuda(), wl["state"].cuda()
    cs, st = cs0.clone(), s0.clone()
    out = torch.empty((4, Hv, D), device="cuda", dtype=torch.float16)
    y3 = torch.empty((3, C), device="cuda", dtype=torch.float16)
    cu3 = gi.cu_seqlens([3]).cuda()
    qk = Hk * D
    stream = torch.cuda.current_stream()

    def four():
        for t in range(4):
            gdn.gdn_decode_step(d, xs[t:t + 1], a[t:t + 1], b[t:t + 1], dp, dt, cw, cs, st,
                                z=z[t:t + 1], norm_w=nw, out=out[t:t + 1])

    def multi():
        gdn.gdn_decode_multi(d, xs.view(1, 4, C), a.view(1, 4, Hv), b.view(1, 4, Hv), dp, dt, cw,
                             cs, st, z=z.view(1, 4, Hv, D), norm_w=nw, out=out.view(1, 4, Hv, D))

    def split():
        gdn.gdn_conv_update(d, cu3, xs[:3], cw, cs, y3)
        gdn.gdn_prefill_chunked(d, cu3, y3[:, :qk], y3[:, qk:2 * qk], y3[:, 2 * qk:], a[:3], b[:3],
                                dp, dt, st, z=z[:3], norm_w=nw, out=out[:3])
        gdn.gdn_decode_step(d, xs[3:], a[3:], b[3:], dp, dt, cw, cs, st, z=z[3:], norm_w=nw,
                            out=out[3:])

    def timed(fn, reps=20):
        for _ in range(3):
            cs.copy_(cs0)
            st.copy_(s0)
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            cs.copy_(cs0)
            st.copy_(s0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(ts)

    t_four, t_multi, t_split = timed(four), timed(multi), timed(split)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            four()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    t_graph = timed(g.replay)
    state_bytes = 2 * Hv * D * D * 4
    return {"workload": "batch-1 layer, 4 tokens: Hk=16 Hv=32 D=128, Grouped, log-rate, f16 "
                        "activations, fp32 state, fused gated norm",
            "unit": "us",
            "four_decode_steps_us": round(_barrier_max(t_four, ws) * 1e6, 2),
            "four_decode_steps_graph_us": round(_barrier_max(t_graph, ws) * 1e6, 2),
            "decode_multi_4_tokens_us": round(_barrier_max(t_multi, ws) * 1e6, 2),
            "split_3_plus_1_us": round(_barrier_max(t_split, ws) * 1e6, 2),
            "us_per_token_graph": round(_barrier_max(t_graph, ws) * 1e6 / 4, 2),
            "state_bytes_per_token": state_bytes,
            "timing": "median of 20 passes between CUDA events, states reset before each; the "
                      "split pass is conv update + chunked prefill (3 tokens, the single-pass "
                      "kernel for f16) + one decode step"}


def run_decode_layer(args, ws, peaks):
    """The whole decode layer on synthetic bf16 weights (gdn_decode_layer:
    fused input projection, decode step with gated RMSNorm, output
    projection): Hk=16, Hv=32, D=128, hidden 2048, Grouped, log-rate, at
    B=64 and B=1. Weight and state sets are cycled so that each step's
    bytes are not in L2 from the step before (sets x (weights + state) >=
    256 MB); the K steps run as one CUDA graph. The two projections are also
    timed alone (gdn_linear, same cycling) for their weight-streaming rate."""
    import gated_delta_net_causal_gb300 as gdn
    Hk, Hv, D, hidden = 16, 32, 128, 2048
    shape = gi.Shape(Hk, Hv, D, map=gi.GROUPED, decay=gi.LOG_RATE, dtype="bf16")
    C, vw = shape.qkv_features, Hv * D
    n_in = (C + vw + 2 * Hv + 63) // 64 * 64
    d = gdn.dims(Hk, Hv, D, map=shape.map, decay=shape.decay, io_dtype=torch.bfloat16)
    g = gi.rng(gi.SEED_BASE + 77)
    wts = gi.layer_weights(g, shape)
    cw, dp, dt, nw = (getattr(wts, n).cuda() for n in ("conv_w", "decay_param", "dt_bias", "norm_w"))
    w_bytes = (n_in * hidden + hidden * vw) * 2
    stream = torch.cuda.current_stream()
    res = {"workload": "decode layer on synthetic bf16 weights: hidden 2048, Hk=16 Hv=32 D=128, "
                       "Grouped, log-rate; fused qkv|z|b|a projection, decode step with gated "
                       "RMSNorm, output projection",
           "unit": "us per layer step", "weight_bytes": w_bytes}
    for B in (64, 1):
        state_b = B * Hv * D * D * 4
        nsets = max(2, -(-256 * 2**20 // (w_bytes + state_b)))
        sets = []
        for _ in range(nsets):
            sets.append(dict(
                w_in=gi.to_dtype(gi.normal(g, (n_in, hidden), hidden ** -0.5), "bf16").cuda(),
                w_out=gi.to_dtype(gi.normal(g, (hidden, vw), vw ** -0.5), "bf16").cuda(),
                cs=gi.to_dtype(gi.normal(g, (B, C, 3), 0.1), "bf16").cuda(),
                st=gi.delta_state(g, shape, B, std=0.02).cuda()))
        xs = [gi.to_dtype(gi.normal(g, (B, hidden), 1.0), "bf16").cuda() for _ in range(4)]
        y = torch.empty((B, hidden), device="cuda", dtype=torch.bfloat16)
        wsb = torch.empty(gdn.gdn_decode_layer_workspace_size(d, hidden, B), device="cuda",
                          dtype=torch.uint8)
        lin_ws = torch.empty(max(gdn.gdn_linear_workspace_size(B, n_in, hidden),
                                 gdn.gdn_linear_workspace_size(B, hidden, vw)), device="cuda",
                             dtype=torch.uint8)
        proj = torch.empty((B, n_in), device="cuda", dtype=torch.bfloat16)
        yc = torch.empty((B, vw), device="cuda", dtype=torch.bfloat16)

        def step(i):
            st = sets[i % nsets]
            gdn.gdn_decode_layer(d, xs[i % 4], st["w_in"], st["w_out"], cw, dp, dt, nw, st["cs"],
                                 st["st"], y, workspace=wsb)

        def lin_in(i):
            gdn.gdn_linear(xs[i % 4], sets[i % nsets]["w_in"], proj, workspace=lin_ws)

        def lin_out(i):
            gdn.gdn_linear(yc, sets[i % nsets]["w_out"], y, workspace=lin_ws)

        def graph_time(fn, k=16):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.stream(side):
                with torch.cuda.graph(gr, stream=side):
                    for i in range(k):
                        fn(i)
            stream.wait_stream(side)
            gr.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            return _barrier_max(e0.elapsed_time(e1) * 1e-3 / k, ws)

        t_layer = graph_time(step)
        t_in, t_out = graph_time(lin_in), graph_time(lin_out)
        step_bytes = w_bytes + 2 * state_b + 2 * B * C * 3 * 2
        res[f"B{B}"] = {
            "us_per_step": round(t_layer * 1e6, 2),
            "bytes_per_step": step_bytes,
            "gbs": round(step_bytes / t_layer / 1e9, 1),
            "hbm_frac": round(step_bytes / t_layer / 1e9 / peaks["hbm_gbs"], 4),
            "in_projection_us": round(t_in * 1e6, 2),
            "in_projection_weight_gbs": round(n_in * hidden * 2 / t_in / 1e9, 1),
            "out_projection_us": round(t_out * 1e6, 2),
            "out_projection_weight_gbs": round(hidden * vw * 2 / t_out / 1e9, 1),
            "launches_per_step": 4, "weight_sets_cycled": nsets,
            "timing": "16 consecutive steps as one CUDA graph replay between two CUDA events"}
        del sets, wsb, lin_ws
        torch.cuda.empty_cache()
    return res


def run_multilayer(args, ws, peaks):
    """Large-batch multi-layer decode: 48 layers back to back on one stream,
    each one token per sequence for B=128 sequences (Hk=16, Hv=48, D=128,
    Grouped, log-rate decay with A_log = ln U[1,16] and dt_bias ~ U(-0.5,
    0.5), bf16 activations ~N(0,1), fp32 states ~N(0,0.02)). Every layer has
    its own state (384 MiB; 18 GiB for the 48), conv state, weights and
    activations, so no layer finds its state in L2; one step = all 48 layers,
    timed with CUDA events on the launching stream."""
    import gated_delta_net_causal_gb300 as gdn
    nl, B, Hk, Hv, D = 48, 128, 16, 48, 128
    C = (2 * Hk + Hv) * D
    gen = torch.Generator(device="cuda").manual_seed(gi.SEED_BASE + 2)
    bf = torch.bfloat16

    def rn(*shape, std=1.0, dtype=bf):
        return (torch.randn(shape, device="cuda", generator=gen) * std).to(dtype)
    d = gdn.dims(Hk, Hv, D, map=gdn.GDN_MAP_GROUPED, decay=gdn.GDN_DECAY_LOG_RATE, io_dtype=bf)
    nw = (0.82 + 0.013 * torch.arange(D, device="cuda")).float()
    layers = []
    for _ in range(nl):
        layers.append({
            "state": rn(B, Hv, D, D, std=0.02, dtype=torch.float32), "cs": rn(B, C, 3, std=0.1),
            "w": rn(C, 4, std=0.16),
            "dp": torch.log(torch.rand(Hv, device="cuda", generator=gen) * 15 + 1),
            "dt": torch.rand(Hv, device="cuda", generator=gen) - 0.5,
            "x": rn(B, C), "a": rn(B, Hv), "b": rn(B, Hv), "z": rn(B, Hv, D),
            "out": torch.empty((B, Hv, D), device="cuda", dtype=bf)})
    stream = torch.cuda.current_stream()

    def step():
        for L in layers:
            gdn.gdn_decode_step(d, L["x"], L["a"], L["b"], L["dp"], L["dt"], L["w"], L["cs"],
                                L["state"], z=L["z"], norm_w=nw, out=L["out"])

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    # the 48 layers of one step as one CUDA graph, replayed per step
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    n = 5
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        ev[i][0].record(stream)
        graph.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    del graph
    t = _barrier_max(statistics.mean(a.elapsed_time(b) * 1e-3 for a, b in ev), ws)
    state_bytes = 2 * nl * B * Hv * D * D * 4
    gbs = ws * state_bytes / t / 1e9
    del layers
    torch.cuda.empty_cache()
    return {"workload": "multi-layer decode: 48 layers x B=128 x 1 token back to back, Hk=16 "
                        "Hv=48 D=128, Grouped, log-rate, bf16 activations, fp32 states (18 GiB)",
            "value": round(gbs, 2), "unit": "GB/s", "metric": "decode state GB/s",
            "ms_per_step": round(t * 1e3, 4), "hbm_frac_state": round(gbs / ws / peaks["hbm_gbs"], 4),
            "us_per_layer": round(t * 1e6 / nl, 2), "launches_per_step": nl,
            "timing": "one step = the 48 layer launches as one CUDA graph replay between two "
                      "CUDA events; mean of 5 steps after 2 eager steps and one replay",
            "l2": "inputs larger than L2 (each layer's state 384 MiB)"}


def run_multi_decode(args, ws, peaks, T=4):
    """The batched-decode shape (B=64, Hk=16, Hv=32, D=128, Tiled,
    negative-rate, bf16) with T=4 tokens per sequence and call
    (gdn_decode_multi: each state read and written once per call). Four state
    sets cycled, the K calls as one CUDA graph, as in the headline. Beside it,
    the route without the call: gdn_conv_update over the B*T tokens then
    gdn_prefill_chunked over B sequences of T tokens (chunk-parallel path,
    workspace allocated once), timed the same way."""
    import gated_delta_net_causal_gb300 as gdn
    B, Hk, Hv, D = 64, 16, 32, 128
    _, d, dev, steps, host, state, cstate, out1, shape = _decode_setup(B, 16, 0)
    del host
    C = shape.qkv_features
    gen = torch.Generator(device="cuda").manual_seed(gi.SEED_BASE + 7)
    bf = torch.bfloat16

    def rn(*sh, std=1.0):
        return (torch.randn(sh, device="cuda", generator=gen) * std).to(bf)
    inputs = [{"x": rn(B, T, C), "a": rn(B, T, Hv), "b": rn(B, T, Hv), "z": rn(B, T, Hv, D)}
              for _ in range(4)]
    nsets = max(4, -(-512 * 2**20 // state.nbytes))
    states = [state] + [state.clone() for _ in range(nsets - 1)]
    cstates = [cstate] + [cstate.clone() for _ in range(nsets - 1)]
    out = torch.empty((B, T, Hv, D), device="cuda", dtype=bf)
    stream = torch.cuda.current_stream()

    def mstep(i):
        x = inputs[i % 4]
        gdn.gdn_decode_multi(d, x["x"], x["a"], x["b"], dev["decay_param"], dev["dt_bias"],
                             dev["conv_w"], cstates[i % nsets], states[i % nsets], z=x["z"],
                             norm_w=dev["norm_w"], out=out)

    # the prefill route over the same tokens: packed [B*T] rows, cu_seqlens of T
    cu = torch.arange(0, B * T + 1, T, device="cuda", dtype=torch.int32)
    y = torch.empty((B * T, C), device="cuda", dtype=bf)
    wsb = torch.empty(gdn.gdn_prefill_workspace_size(d, B, B * T), device="cuda",
                      dtype=torch.uint8)
    qk = Hk * D

    def pstep(i):
        x = inputs[i % 4]
        cs, st = cstates[i % nsets], states[i % nsets]
        gdn.gdn_conv_update(d, cu, x["x"].view(B * T, C), dev["conv_w"], cs, y)
        gdn.gdn_prefill_chunked(d, cu, y[:, :qk], y[:, qk:2 * qk], y[:, 2 * qk:],
                                x["a"].view(B * T, Hv), x["b"].view(B * T, Hv),
                                dev["decay_param"], dev["dt_bias"], st, z=x["z"].view(B * T, Hv, D),
                                norm_w=dev["norm_w"], out=out.view(B * T, Hv, D), workspace=wsb)

    def timed(fn, graphed=True):
        for i in range(max(args.warmup, 4)):
            fn(i)
        torch.cuda.synchronize()
        if not graphed:
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for i in range(args.steps):
                fn(i)
            ev1.record(stream)
            torch.cuda.synchronize()
            return _barrier_max(ev0.elapsed_time(ev1) * 1e-3 / args.steps, ws)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                for i in range(args.steps):
                    fn(i)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        graph.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        del graph
        return _barrier_max(ev0.elapsed_time(ev1) * 1e-3 / args.steps, ws)

    t_multi = timed(mstep)
    t_pref = timed(pstep, graphed=False)
    del states, cstates, inputs, wsb
    torch.cuda.empty_cache()
    state_bytes = 2 * B * Hv * D * D * 4
    return {"workload": f"multi-token decode: B=64 sequences x {T} tokens per call, Hk=16 Hv=32 "
                        "D=128, Tiled, negative-rate, bf16",
            "value": round(ws * B * T / t_multi, 1), "unit": "tokens/s",
            "ms_per_call": round(t_multi * 1e3, 5),
            "state_gbs": round(ws * state_bytes / t_multi / 1e9, 2),
            "hbm_frac_state": round(state_bytes / t_multi / 1e9 / peaks["hbm_gbs"], 4),
            "via_conv_and_prefill_ms": round(t_pref * 1e3, 5),
            "via_conv_and_prefill_timing": "gdn_conv_update + gdn_prefill_chunked per call, "
                                           "issued eagerly back to back (five launches)",
            "l2": f"inputs larger than L2: {nsets} state sets cycled",
            "timing": f"the {args.steps} consecutive calls as one CUDA graph replay"}


def run_slot_decode(args, ws, peaks):
    """The batched-decode shape (B=64, Hk=16, Hv=32, D=128, Tiled,
    negative-rate, bf16) through gdn_decode_step_slots: the 64 rows name
    slots of a pool of 256 states (fp32 ~N(0, 0.02), 512 MiB). Four slot
    tables, one seeded permutation of the pool cut in four, are cycled step
    by step, so a step's states were last touched four steps earlier (inputs
    larger than L2). Timed like the headline: the K steps as one CUDA graph."""
    import gated_delta_net_causal_gb300 as gdn
    B, P, Hv, D = 64, 256, 32, 128
    gdn_, d, dev, steps, host, state, cstate, out, shape = _decode_setup(B, 16, 0)
    del host, state, cstate
    gen = torch.Generator(device="cuda").manual_seed(gi.SEED_BASE + 6)
    pool = torch.randn((P, Hv, D, D), device="cuda", generator=gen) * 0.02
    cpool = (torch.randn((P, shape.qkv_features, 3), device="cuda", generator=gen) * 0.1).to(
        torch.bfloat16)
    perm = torch.randperm(P, device="cuda", generator=gen).to(torch.int32)
    tables = [perm[i * B:(i + 1) * B].contiguous() for i in range(P // B)]
    stream = torch.cuda.current_stream()

    def step(i):
        inp = steps[i % 16]
        gdn.gdn_decode_step_slots(d, tables[i % len(tables)], inp["x"], inp["a"], inp["b"],
                                  dev["decay_param"], dev["dt_bias"], dev["conv_w"], cpool, pool,
                                  z=inp["z"], norm_w=dev["norm_w"], out=out)

    for i in range(max(args.warmup, 4)):
        step(i)
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(args.steps):
                step(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    graph.replay()
    ev1.record(stream)
    torch.cuda.synchronize()
    t = _barrier_max(ev0.elapsed_time(ev1) * 1e-3 / args.steps, ws)
    del graph, pool, cpool
    torch.cuda.empty_cache()
    state_bytes = 2 * B * Hv * D * D * 4
    gbs = ws * state_bytes / t / 1e9
    return {"workload": "batched decode through a state-slot table: B=64 rows in a pool of 256 "
                        "slots, Hk=16 Hv=32 D=128, Tiled, negative-rate, bf16",
            "value": round(gbs, 2), "unit": "GB/s", "metric": "decode state GB/s",
            "ms_per_step": round(t * 1e3, 5),
            "hbm_frac_state": round(gbs / ws / peaks["hbm_gbs"], 4),
            "l2": "inputs larger than L2: four disjoint slot tables of 64 cycled (512 MiB pool)",
            "timing": f"the {args.steps} consecutive steps as one CUDA graph replay"}


# --------------------------------------------------------------- CPU oracle arm

def cpu_baseline_decode(seconds: float = 15.0, threads: int = None):
    """The oracle (as it stands) on a bounded sample of the decode workload:
    repeated decode steps over a subset of the B=64 sequences, one sequence
    per host thread (ctypes releases the GIL inside the C oracle)."""
    import concurrent.futures as cf
    import oracle
    threads = threads or min(os.cpu_count() or 1, 64)
    wl = gi.workload_batched_decode(batch=64, sets=2)
    shape, w = wl["shape"], wl["weights"]
    F = gi.as_f64
    cw, dp, dt, nw = F(w.conv_w), F(w.decay_param), F(w.dt_bias), F(w.norm_w)
    seqs = list(range(min(threads, 64)))
    X = [F(s.mixed_qkv) for s in wl["steps"]]
    A = [F(s.a) for s in wl["steps"]]
    Bb = [F(s.b) for s in wl["steps"]]
    Z = [F(s.z) for s in wl["steps"]]
    cs = {b: F(wl["conv_state"])[b] for b in seqs}
    S = {b: F(wl["state"])[b] for b in seqs}

    def one(b, i):
        _, _, cs[b], S[b] = oracle.segment(16, 32, 128, shape.map, shape.decay,
                                           X[i % 2][b:b + 1], A[i % 2][b:b + 1],
                                           Bb[i % 2][b:b + 1], Z[i % 2][b:b + 1], cw, dp, dt,
                                           nw, cs[b], S[b])

    oracle.lib()
    done = 0
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=len(seqs)) as ex:
        i = 0
        while time.perf_counter() - t0 < seconds or i == 0:
            list(ex.map(lambda b: one(b, i), seqs))
            done += len(seqs)
            i += 1
    el = time.perf_counter() - t0
    bytes_per_seq = 2 * 32 * 128 * 128 * 4
    return {"value": round(done * bytes_per_seq / el / 1e9, 4), "unit": "GB/s",
            "cores": len(seqs), "kind": "oracle",
            "sample": f"{i} decode steps x {len(seqs)} of the 64 sequences (fp64 oracle, "
                      f"one sequence per thread), {el:.1f} s"}


def cpu_baseline_prefill(wl, seconds: float = 15.0, threads: int = None):
    """The oracle (as it stands) on the T=4096 prefill workload: the l2 norms,
    gates and the token recurrence of every V head over the first tokens of
    the sequence (one head per host thread, ctypes releases the GIL inside the
    C oracle), repeated over growing token counts until about `seconds` have
    passed; the rate is tokens of the whole layer (all 32 V heads) per
    second."""
    import concurrent.futures as cf
    import oracle
    F = gi.as_f64
    shape, w = wl["shape"], wl["weights"]
    threads = threads or min(os.cpu_count() or 1, 32)
    gg, bb = oracle.gates(F(wl["a"]), F(wl["b"]), F(w.decay_param), F(w.dt_bias), shape.decay)
    q = oracle.l2norm(F(wl["q"]))
    k = oracle.l2norm(F(wl["k"]))
    v = F(wl["v"])
    S0 = F(wl["state"])[0]
    Hk, Hv = shape.n_k_heads, shape.n_v_heads

    def head(args_):
        h, T_s = args_
        kh = oracle.k_head(shape.map, h, Hk, Hv)
        oracle.delta(q[:T_s, kh:kh + 1], k[:T_s, kh:kh + 1], v[:T_s, h:h + 1], gg[:T_s, h:h + 1],
                     bb[:T_s, h:h + 1], S0[h:h + 1], 0)

    oracle.lib()
    tokens = 0
    T_s = 256
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while True:
            list(ex.map(head, [(h, T_s) for h in range(Hv)]))
            tokens += T_s
            if time.perf_counter() - t0 >= seconds:
                break
            T_s = min(2 * T_s, 4096)
    el = time.perf_counter() - t0
    return {"value": round(tokens / el, 2), "unit": "tokens/s", "cores": threads, "kind": "oracle",
            "sample": f"the token recurrence of all {Hv} V heads over {tokens} tokens in total "
                      f"(prefixes of the T=4096 sequence, fp64 oracle, one head per thread), "
                      f"{el:.1f} s"}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    cb = cpu_baseline_decode(seconds=max(5.0, min(60.0, args.cpu_seconds)))
    return {"impl": "reference",
            "metric": "GDN decode state GB/s (% HBM peak); chunked prefill tokens/s (% roofline)",
            "value": cb["value"], "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DECODE_WORKLOAD, "global_batch": 64},
            "cpu_baseline": cb,
            "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--batch", type=int, default=64)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-multilayer", action="store_true", help="skip the 48-layer decode block")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the state-slot and multi-token decode blocks")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the T=4096 chunked-prefill block (a process of about 1.5 GB "
                         "on the device, for profiler captures of the prefill kernels)")
    ap.add_argument("--only", default=None,
                    choices=["prefill", "varlen_path", "decode_layer", "multi_token_decode",
                             "slot_decode"],
                    help="run only this block and print it (for profiler captures of its kernels)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "gb300" else "gloo")
    try:
        if args.impl == "reference":
            line = run_reference(args, ws, rank)
        else:
            line = run_gpu(args, ws, rank, local)
        if line is not None:
            print(json.dumps(line), flush=True)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
