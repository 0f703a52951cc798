"""Host logic of bench.py on CPU (no GPU): the clock-sample summary and its window, the
DRAM-traffic figures keyed by the kernels' source hashes, the workload configs the JSON
line carries, and one short run of the reference arm (the float64 oracle on the host
cores) with the keys of its JSON line."""
import json
import os
import subprocess
import sys

import pytest

import bench
from workloads import CAUSAL_D256_FWD_BWD, CAUSAL_FWD_BWD, CAUSAL_FWD_BWD_DROPOUT

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sampler(lines, first=0, last=None):
    c = bench.ClockSampler(0)
    c.lines = list(lines)
    c.first, c.last = first, len(lines) if last is None else last
    return c


def test_clock_summary_median_max_and_reasons():
    lines = ["2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
             "2055, 2070, 1350.0, Not Active, Not Active, Not Active, Active",
             "2070, 2070, 1390.2, Not Active, Not Active, Not Active, Active"]
    s = _sampler(lines).summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"],
                 "samples": 3}
    hot = _sampler(["1800, 2070, 1400, Active, Not Active, Active, Not Active"]).summary()
    assert hot["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_counts_only_the_timed_window():
    lines = ["1000, 2070, 100, Not Active, Not Active, Not Active, Not Active",  # before
             "2070, 2070, 900, Not Active, Not Active, Not Active, Not Active",
             "2070, 2070, 900, Not Active, Not Active, Not Active, Not Active",
             "1200, 2070, 100, Active, Not Active, Not Active, Not Active"]     # after
    s = _sampler(lines, first=1, last=3).summary()
    assert s["samples"] == 2 and s["sm_mhz"] == 2070.0 and s["reasons"] == []
    empty = _sampler(lines, first=4, last=4).summary()
    assert empty["samples"] == 0 and empty["reasons"] == ["unsampled"]
    bad = _sampler(["[N/A], [N/A], x"]).summary()
    assert bad["samples"] == 0


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    sha = bench.kernel_source_sha("dkdv_kernel")
    monkeypatch.setitem(bench.NCU_TRAFFIC, "dkdv_kernel", {"bytes": 123, "sha256": sha})
    assert bench.ncu_traffic("dkdv_kernel") == 123
    monkeypatch.setitem(bench.NCU_TRAFFIC, "dkdv_kernel", {"bytes": 123, "sha256": "0" * 64})
    assert bench.ncu_traffic("dkdv_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None
    # every kernel named in the table hashes files that exist
    for k in bench.NCU_TRAFFIC:
        assert len(bench.kernel_source_sha(k)) == 64


def test_workload_configs():
    c = bench.workload_config(CAUSAL_FWD_BWD, {"parallelism": "replicas x1"})
    assert c["N"] == 8192 and c["d"] == 128 and c["mask"] == "causal"
    assert "dropout_p" not in c and c["parallelism"] == "replicas x1"
    c = bench.workload_config(CAUSAL_FWD_BWD_DROPOUT)
    assert c["dropout_p"] == 0.1 and c["dropout_seed"] >> 32 and c["dropout_seed"] & 0xFFFFFFFF
    c = bench.workload_config(CAUSAL_D256_FWD_BWD)
    assert c["d"] == 256 and "inputs 512 MiB" in c["l2"]


def test_reference_arm_line():
    """`bench.py --impl reference` times the oracle on one head per step."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "dtype", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC


def _bench(*argv, env=None, timeout=600):
    e = dict(os.environ)
    for key in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        e.pop(key, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv],
                          capture_output=True, text=True, timeout=timeout, cwd=ROOT, env=e)


def test_gpus_n_launches_n_replicas():
    """`bench.py --gpus 2` started without a launcher starts two ranks itself (the same
    torch.distributed.run entry the driver uses); the line reports n_gpus 2, the job time
    is the slower rank's and the value sums both replicas' work over it. The step is the
    CPU check workload (gloo ranks, no GPU)."""
    r = _bench("--gpus", "2", "--workload", "cpu_replica_check", "--steps", "20",
               "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["config"]["parallelism"] == "replicas x2"
    work = 2.0 * 256 ** 3 * 20
    ms_total = line["ms_per_step"] * 20
    assert ms_total >= line["rank0_ms"] - 1e-4          # max over ranks (6-digit rounding)
    assert abs(line["value"] - 2 * work / (ms_total * 1e-3) / 1e9) <= 1e-3 * line["value"]


def test_world_size_must_match_gpus():
    r = _bench("--gpus", "2", "--workload", "cpu_replica_check",
               env={"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr


def test_repeat_timed_covers_min_seconds(monkeypatch):
    """The timed region (K steps) is repeated until its GPU time reaches --min-seconds."""
    import types

    class Quiet:
        def __init__(self, index):
            pass

        def __enter__(self):
            return self

        def __exit__(self, *exc):
            pass

        def summary(self):
            return {"samples": 0}

    monkeypatch.setattr(bench, "ClockSampler", Quiet)
    calls = []

    def rep():  # 4 steps of 3 kernels, 25 ms per step
        calls.append(1)
        return [[10.0, 5.0, 10.0] for _ in range(4)]

    args = types.SimpleNamespace(min_seconds=1.0, steps=4)
    rows, n, _ = bench.repeat_timed(args, 1, types.SimpleNamespace(index=0), rep)
    assert n == 10 and len(calls) == 10 and len(rows) == 40  # 10 x 100 ms >= 1 s
    args.min_seconds = 0.0
    rows, n, _ = bench.repeat_timed(args, 1, types.SimpleNamespace(index=0), rep)
    assert n == 1 and len(rows) == 4


def test_reference_arm_follows_the_workload():
    """The reference arm of a forward-only workload times the oracle's forward on blocks
    of query rows, with the forward metric."""
    r = _bench("--impl", "reference", "--workload", "tiny_fwd", "--steps", "2", "--warmup", "1")
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["steps"] == 2
    assert line["metric"].startswith("attention forward TFLOP/s")
    assert "query rows" in line["cpu_baseline"]["sample"]


def test_roofline_peak_follows_the_timed_region():
    """A timed region of a second or more is a sustained measurement under the power cap:
    its tensor roofline takes the sustained bf16 figure; a short burst takes the burst one."""
    pk = {"bf16_tflops": 1908.0, "bf16_sustained": 1728.7, "hbm_gbs": 6744.6}
    assert bench.tensor_peak(pk, 2000.0) == (1728.7, "bf16 sustained (timed region >= 1 s)")
    assert bench.tensor_peak(pk, 35.0) == (1908.0, "bf16 burst")
