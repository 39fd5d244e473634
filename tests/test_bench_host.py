"""Host-side logic of bench.py, without a GPU: the profile gate on the
roofline's DRAM traffic, the peaks it divides by, the oracle's CPU-baseline
sample and the reference arm's JSON line."""

import argparse
import json
import os

import bench


def test_kernel_hash_is_stable_and_short():
    a = bench._kernel_hash("decode.cu", "gdn_common.cuh")
    assert a == bench._kernel_hash("decode.cu", "gdn_common.cuh")
    assert len(a) == 16 and int(a, 16) >= 0
    assert a != bench._kernel_hash("decode_mt.cu", "gdn_common.cuh")


def test_profile_traffic_only_for_the_profiled_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    (tmp_path / "k.txt").write_text("# a comment = ignored\nkernel_hash = abc\n"
                                    "dram_bytes_per_launch = 1234\n")
    assert bench._profile_traffic("k.txt", "abc") == 1234.0
    assert bench._profile_traffic("k.txt", "abd") is None  # source changed since
    assert bench._profile_traffic("missing.txt", "abc") is None


def test_committed_profiles_parse():
    for name in ("decode_step_b64.txt", "prefill_cp_t4096.txt"):
        kv = {}
        with open(os.path.join(bench.PROFILES, name)) as f:
            for line in f:
                if "=" in line and not line.lstrip().startswith("#"):
                    k, v = line.split("=", 1)
                    kv[k.strip()] = v.strip()
        assert len(kv["kernel_hash"]) == 16
        assert float(kv["dram_bytes_per_launch"]) > 1e8


def test_peaks_come_from_the_measured_file():
    pk = bench._peaks()
    if os.path.exists(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")):
        assert pk["source"] == "measured"
        with open(os.path.join(bench.ROOT, "MEASURED_PEAKS.json")) as f:
            assert pk["hbm_gbs"] == float(json.load(f)["hbm_gbs"])
    assert pk["hbm_gbs"] > 1000 and pk["bf16_tflops"] > 100


def test_cpu_baseline_sample_is_bounded_and_described():
    cb = bench.cpu_baseline_decode(seconds=0.05, threads=2)
    assert cb["kind"] == "oracle" and cb["cores"] == 2 and cb["unit"] == "GB/s"
    assert cb["value"] > 0 and "decode steps" in cb["sample"]


def test_reference_line_contract(monkeypatch):
    fake = {"value": 1.5, "unit": "GB/s", "cores": 3, "kind": "oracle", "sample": "s"}
    monkeypatch.setattr(bench, "cpu_baseline_decode", lambda seconds: fake)
    args = argparse.Namespace(steps=7, warmup=3, cpu_seconds=0.1)
    line = bench.run_reference(args, 1, 0)
    json.dumps(line)
    assert line["impl"] == "reference" and line["value"] == 1.5 and line["unit"] == "GB/s"
    assert line["higher_is_better"] is True and line["steps"] == 7 and line["warmup"] == 3
    assert line["cpu_baseline"] == fake
    assert line["e2e"] == {"value": 1.5, "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == bench.DECODE_WORKLOAD
