"""Benchmark: one step = the whole hot path (tile classification, forward with the
online softmax, backward rebuilding P from the LSE) on the causal fwd+bwd workload
(B=2, H=16, N=8192, d=128, bf16), timed with CUDA events.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--min-seconds S]
                [--workload fwd_bwd|fwd_bwd_dropout|fwd_bwd_d256|causal_fwd|gqa_window_fwd
                            |docs_fwd|tiny_fwd|fp8_causal_fwd|causal_fwd_d256|paged_decode
                            |cpu_replica_check]

Prints one JSON line. `value` is useful TFLOP/s (masked-out work excluded) summed
over ranks; with N > 1 each rank runs its own replica of the workload (the heads
are independent, so there is no data-path collective). Launched under
torch.distributed.run, the ranks come from its environment; `--gpus N` given alone
starts the N ranks itself the same way (127.0.0.1 rendezvous, one GPU per rank).
The timed region, exactly K steps between a barrier and a device synchronisation
on both sides, is repeated until the repetitions cover at least --min-seconds of
GPU time (default 2 s), so that the clock samplers see the kernels under load; the
line reports the mean per step over all repetitions and how many there were.
--impl reference times the float64 CPU oracle on a bounded sample of the same
workload on the host cores. cpu_replica_check runs the launcher and the cross-rank
reduction on CPU (gloo ranks, a float64 matmul as the step); the tests use it.
--workload picks one of the other workloads: fwd_bwd_dropout and fwd_bwd_d256 are the
fwd+bwd step with dropout p = 0.1 and at head dimension 256; the *_fwd ones are
forward-only, so a step is one forward pass and the line reports the forward's useful
TFLOP/s. fp8_causal_fwd
runs the FP8 forward (e4m3 inputs with block scales, quantised once before the timed
steps; the end-to-end number includes the quantisation). paged_decode times one decode
step over a paged KV cache and reports GB/s against the HBM roofline.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import (CAUSAL, CAUSAL_D256, CAUSAL_D256_FWD_BWD, CAUSAL_FWD_BWD,  # noqa: E402
                       CAUSAL_FWD_BWD_DROPOUT, DOCS, GQA_WINDOW, MASK_NAMES, PAGED_DECODE, TINY, make_decode_inputs, make_inputs)

FWD_WORKLOADS = {"causal_fwd": CAUSAL, "gqa_window_fwd": GQA_WINDOW, "docs_fwd": DOCS,
                 "tiny_fwd": TINY, "fp8_causal_fwd": CAUSAL, "causal_fwd_d256": CAUSAL_D256}

METRIC = "attention fwd/bwd TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 peak"
UNIT = "TFLOP/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        return {"bf16_tflops": m["bf16_tflops"], "bf16_sustained": m["bf16_tflops_sustained"],
                "hbm_gbs": m["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def tensor_peak(pk, gpu_ms: float):
    """The bf16 tensor peak a kernel's roofline fraction is taken against: the sustained
    figure (a seconds-long loop under the power cap) when the timed region covers at
    least a second of GPU time, as it does by default, else the burst figure."""
    if gpu_ms >= 1000.0:
        return pk["bf16_sustained"], "bf16 sustained (timed region >= 1 s)"
    return pk["bf16_tflops"], "bf16 burst"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines: list[str] = []
        self.first = self.last = 0

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # let nvidia-smi start (up to 3 s), then count only what comes after
            t_end = time.perf_counter() + 3.0
            while not self.lines and time.perf_counter() < t_end:
                time.sleep(0.01)
        except (OSError, ValueError):
            self.proc = None
        self.first = len(self.lines)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        self.last = len(self.lines)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines[self.first:self.last]:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, flag in zip(names, parts[3:7]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# DRAM bytes (read + write) per launch from one ncu capture of each kernel on this
# workload, keyed by the SHA-256 of the kernel's sources (its .cu file plus the shared
# headers) at capture time. A kernel whose sources have changed since reports null.
KERNEL_SOURCES = {"fwd_tc_kernel": ("fwd_tc.cu",), "dkdv_kernel": ("bwd_tc.cu", "bwd_common.cuh"),
                  "dq_kernel": ("bwd_tc.cu", "bwd_common.cuh"), "rowdot_kernel": ("simt.cu",),
                  "decode_tc_kernel": ("decode_tc.cuh", "decode_tc.cu", "decode_copies2.cu")}
SHARED_HEADERS = ("ptx.cuh", "mask.cuh", "kernels.h")
# decode_tc_kernel: the paged-decode workload (B=64, lengths 512-8192).
NCU_TRAFFIC = {
    "fwd_tc_kernel": {"bytes": 201466112 + 47017728,
                    "sha256": "a1501cbbd8b5048f95c2734dbc48c13a2eb13f54bc772e83e29c3bd13d491c1a"},
    "rowdot_kernel": {"bytes": 135310080 + 485888,
                    "sha256": "907130b51cc9542e5c71b7061ffeb7e26f7e76fde0a5700ed4eb6351009ceb8e"},
    "dkdv_kernel": {"bytes": 270685440 + 101813760,
                  "sha256": "526940b6bb4d74aa8715e5e80f5891713689e090d95e518855f0cf99c8c2d535"},
    "dq_kernel": {"bytes": 270654208 + 49328640,
                "sha256": "526940b6bb4d74aa8715e5e80f5891713689e090d95e518855f0cf99c8c2d535"},
    "decode_tc_kernel": {"bytes": 1119356160 + 9067520,
                       "sha256": "e5baa6b786d411da95b06bbe6b9f34436a88ad59aaa68a53ecd64ab8a0bbfa26"},
}

def kernel_source_sha(kernel: str) -> str:
    """SHA-256 of the kernel's sources with // comments and blank space removed, so that
    an edit of the comments alone keeps the figures of the unchanged code."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_io_aware_13_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel] + SHARED_HEADERS:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = re.sub(r"//[^\n]*", "", f.read())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()


def ncu_traffic(kernel: str):
    entry = NCU_TRAFFIC.get(kernel)
    if not entry:
        return None
    try:
        return entry["bytes"] if kernel_source_sha(kernel) == entry["sha256"] else None
    except OSError:
        return None


def max_over_ranks(x: float, device) -> float:
    """Largest x over all ranks (the job's time is its slowest replica's)."""
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def check_world(args, world: int) -> None:
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}: give --gpus N "
                         "alone, or launch N ranks with torch.distributed.run and --gpus N")


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_replicas(n: int, argv) -> int:
    """`--gpus N` (N > 1) without a launcher: start N ranks of this script through
    torch.distributed.run (one process per GPU, 127.0.0.1 rendezvous). Every rank runs
    its own replica of the workload; rank 0 prints the line. Returns the exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr", "127.0.0.1",
           "--master-port", str(free_port()), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def init_ranks(args, backend: str = "nccl"):
    """(world, rank, local rank) from the launcher's environment, checked against
    --gpus; joins the process group when there is more than one rank."""
    world, rank, local = dist_env()
    check_world(args, world)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return world, rank, local


def repeat_timed(args, world: int, dev, rep):
    """Run `rep` (one timed region of exactly args.steps steps, bracketed by a barrier and
    a synchronisation; it returns one list of kernel times in ms per step) until the
    repetitions cover at least args.min_seconds of GPU time, with the clocks sampled
    throughout. Every rank runs the same number of repetitions (the maximum of the
    ranks' estimates). Returns (rows of all repetitions, repetitions, clock summary)."""
    import math
    with ClockSampler(dev.index if dev.index is not None else 0) as clk:
        rows = rep()
        gpu_ms = sum(sum(r) for r in rows)
        n = max(1, math.ceil(args.min_seconds * 1e3 / max(gpu_ms, 1e-3)))
        if world > 1:
            n = int(max_over_ranks(n, dev))
        for _ in range(n - 1):
            rows += rep()
    return rows, n, clk.summary()


def workload_config(w, extra=None):
    n_in = 4 if w.backward else 3  # q, k, v (and dO)
    mib = (n_in - 2) * w.B * w.Hq * w.Nq * w.d * 2 + 2 * w.B * w.Hkv * w.Nkv * w.d * 2
    cfg = {"workload": w.describe(), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.Nq, "d": w.d,
           "mask": MASK_NAMES[w.mask_kind], "seed": w.seed,
           "l2": f"flushed between steps (256 MiB write); inputs {mib >> 20} MiB"}
    if w.dropout_p > 0:
        cfg.update(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)
    if extra:
        cfg.update(extra)
    return cfg


def pipelined_e2e(steps, stream, dev, host_in, in_sets, out_sets, host_out, run_step):
    """End-to-end time of `steps` steps, ms per step. Step s copies `host_in` (pinned) into
    device input set s % 2, runs `run_step(s % 2)` on the compute stream and copies output
    set s % 2 into `host_out` (pinned). The inputs of step s + 1 arrive and the outputs of
    step s leave on their own streams (one per tensor) while the kernels run; events order
    each copy after the kernels that last used its buffers."""
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s_in_t = [torch.cuda.Stream(device=dev) for _ in host_in]
    s_out_t = [torch.cuda.Stream(device=dev) for _ in host_out]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def fan_out(main, subs, pairs, done):
        start = torch.cuda.Event()
        start.record(main)
        for st_, (dst, src) in zip(subs, pairs):
            st_.wait_event(start)
            with torch.cuda.stream(st_):
                dst.copy_(src, non_blocking=True)
            fin = torch.cuda.Event()
            fin.record(st_)
            main.wait_event(fin)
        done.record(main)

    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    fan_out(s_in, s_in_t, list(zip(in_sets[0], host_in)), ev_in[0])
    for st_i in range(steps):
        x = st_i % 2
        stream.wait_event(ev_in[x])
        if st_i >= 2:
            stream.wait_event(ev_out[x])  # outputs of step st_i - 2 copied out
        run_step(x)
        ev_done[x].record(stream)
        if st_i + 1 < steps:
            if st_i >= 1:
                s_in.wait_event(ev_done[1 - x])  # step st_i - 1 is done with those inputs
            fan_out(s_in, s_in_t, list(zip(in_sets[1 - x], host_in)), ev_in[1 - x])
        s_out.wait_event(ev_done[x])
        fan_out(s_out, s_out_t, list(zip(host_out, out_sets[x])), ev_out[x])
    stream.wait_event(ev_out[(steps - 1) % 2])
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def run_ours(args, w=CAUSAL_FWD_BWD):
    from exact_io_aware_13_gb300 import build as libbuild
    libbuild.build()  # compiles libattn.so from source if it is missing or stale
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import flops
    world, rank, local = init_ranks(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pairs = flops.allowed_pairs(w.mask_kind, w.Nq, w.Nkv)
    f_fwd = flops.attention_flops(w.B, w.Hq, w.d, pairs, backward=False)
    f_bwd = flops.attention_flops(w.B, w.Hq, w.d, pairs, backward=True)
    f_step = f_fwd + f_bwd

    q, k, v, do, _ = make_inputs(w)
    host = [t.pin_memory() for t in (q, k, v, do)]
    qd, kd, vd, dod = (t.to(dev) for t in host)
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:-1], dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(ea.bwd_workspace_size(qd, kd), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kw = dict(scale=w.scale, mask_kind=w.mask_kind)
    if w.dropout_p > 0:
        kw.update(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)

    def step():
        ea.fwd_into(qd, kd, vd, o, lse, **kw)
        ea.bwd_into(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ea.device_status() != 0:
        raise RuntimeError("a kernel gave up a bounded wait during warm-up")

    # ------------------------------------------------------------ device-timed steps
    # Per step: attn_fwd, then the backward's three kernels through attn_bwd_phases
    # (the same launches attn_bwd makes), with an event between kernels so that each
    # kernel's own duration is measured on the stream it runs on.
    # (at d = 256 the dK/dV phase is two kernels, the dV and the dK walk)
    names = (["fwd256_kernel", "rowdot_kernel", "dkdv256_kernel", "dq256_kernel"] if w.d == 256
             else ["fwd_tc_kernel", "rowdot_kernel", "dkdv_kernel", "dq_kernel"])

    def timed_rep():
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for s in range(args.steps):
            flush.zero_()  # evict the previous step's tensors from L2 (untimed)
            ev[s][0].record(stream)
            ea.fwd_into(qd, kd, vd, o, lse, **kw)
            ev[s][1].record(stream)
            for k_, ph in enumerate((ea.BWD_ROWDOT, ea.BWD_DKDV, ea.BWD_DQ)):
                ea.bwd_phases_into(ph, qd, kd, vd, o, lse, dod, dq, dk, dv, ws, **kw)
                ev[s][2 + k_].record(stream)
        torch.cuda.synchronize()
        return [[e[i].elapsed_time(e[i + 1]) for i in range(4)] for e in ev]

    rows, reps, clocks = repeat_timed(args, world, dev, timed_rep)
    if ea.device_status() != 0:
        raise RuntimeError("a kernel gave up a bounded wait during the timed steps")
    n_timed = len(rows)
    per_kernel = {n: [r[i] for r in rows] for i, n in enumerate(names)}
    t_fwd = per_kernel[names[0]]
    t_bwd = [sum(r[1:]) for r in rows]
    t_step = sum(sum(r) for r in rows)  # ms over all timed steps
    if world > 1:
        t_step = max_over_ranks(t_step, dev)
    ms_step = t_step / n_timed
    value = world * f_step / (ms_step * 1e-3) / 1e12

    # ------------------------------------------------------------ end to end, host buffers
    # Every step copies its inputs in from pinned host memory, runs attn_fwd + attn_bwd
    # through the public entry points and copies its results out (pipelined_e2e: two
    # buffer sets, the copies overlap the kernels of the neighbouring steps).
    outs_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                 for t in (o, lse, dq, dk, dv)]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in outs_host)
    in_sets = [(qd, kd, vd, dod), tuple(torch.empty_like(t) for t in (qd, kd, vd, dod))]
    out_sets = [(o, lse, dq, dk, dv), tuple(torch.empty_like(t) for t in (o, lse, dq, dk, dv))]

    def run_step(x):
        (bq, bk, bv, bdo), (bo, blse, bdq, bdk, bdv) = in_sets[x], out_sets[x]
        ea.fwd_into(bq, bk, bv, bo, blse, **kw)
        ea.bwd_into(bq, bk, bv, bo, blse, bdo, bdq, bdk, bdv, ws, **kw)

    if world > 1:
        torch.distributed.barrier()
    ms_e2e = pipelined_e2e(args.steps, stream, dev, host, in_sets, out_sets, outs_host, run_step)
    e2e_value = world * f_step / (ms_e2e * 1e-3) / 1e12

    pk = peaks()
    tpeak, tpeak_name = tensor_peak(pk, sum(sum(r) for r in rows))
    ms_fwd = statistics.mean(t_fwd)
    ms_bwd = statistics.mean(t_bwd)
    fwd_tf = f_fwd / (ms_fwd * 1e-3) / 1e12
    bwd_tf = f_bwd / (ms_bwd * 1e-3) / 1e12
    # Algorithmic work of one launch of each kernel: FLOPs of the
    # contractions it performs per allowed pair, or bytes for the row-dot kernel.
    units = w.B * w.Hq * pairs
    # (d = 256: the dV walk runs S^T and dV, the dK walk S^T, dP^T and dK)
    algo = {names[0]: (4 * w.d * units, "TFLOP/s"),
            names[2]: ((10 if w.d == 256 else 8) * w.d * units, "TFLOP/s"),
            names[3]: (6 * w.d * units, "TFLOP/s"),
            # reads O, dO and L; writes L log2 e and D
            "rowdot_kernel": (w.B * w.Hq * w.Nq * (4 * w.d + 12), "GB/s")}
    kernels = {}
    for n in names:
        ms = statistics.mean(per_kernel[n])
        work, unit = algo[n]
        ach = work / (ms * 1e-3) / (1e12 if unit == "TFLOP/s" else 1e9)
        peak = tpeak if unit == "TFLOP/s" else pk["hbm_gbs"]
        kernels[n] = {"ms": round(ms, 4), "achieved": round(ach, 2), "unit": unit,
                      "frac": round(ach / peak, 4)}
        if unit == "TFLOP/s":
            kernels[n]["frac_of_burst"] = round(ach / pk["bf16_tflops"], 4)
    dom = max(names, key=lambda n: kernels[n]["ms"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded randn rounded to bf16)",
        "config": workload_config(w, {"parallelism": f"replicas x{world}"}),
        "pct_of_peak": round(100 * value / world / pk["bf16_tflops"], 1),
        "fwd": {"tflops": round(fwd_tf, 2), "ms": round(ms_fwd, 4),
                "pct_of_peak": round(100 * fwd_tf / pk["bf16_tflops"], 1)},
        "bwd": {"tflops": round(bwd_tf, 2), "ms": round(ms_bwd, 4),
                "pct_of_peak": round(100 * bwd_tf / pk["bf16_tflops"], 1)},
        "kernels": kernels,
        "roofline": {"bound": "tensor" if algo[dom][1] == "TFLOP/s" else "hbm", "kernel": dom,
                     "achieved": kernels[dom]["achieved"],
                     "peak": tpeak if algo[dom][1] == "TFLOP/s" else pk["hbm_gbs"],
                     "unit": algo[dom][1], "frac": kernels[dom]["frac"],
                     "frac_of_burst": kernels[dom].get("frac_of_burst"),
                     "peak_source": pk["source"] + (" " + tpeak_name if algo[dom][1] == "TFLOP/s"
                                                    else " HBM copy"),
                     # counters were taken on the kernels without dropout
                     "traffic": ncu_traffic(dom) if w.dropout_p == 0 else None},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4)},
        "timed_repeats": reps, "timed_steps": n_timed,
        "gpu_launches": (5 if w.d == 256 else 4) * n_timed,  # d = 256: dV and dK walks
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, seconds=args.cpu_seconds)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_forward(args, w, fp8=False):
    """Forward-only workloads: a step is one attn_fwd (or attn_fwd_fp8) over the whole
    workload."""
    from exact_io_aware_13_gb300 import build as libbuild
    libbuild.build()
    import exact_io_aware_13_gb300 as ea
    from exact_io_aware_13_gb300 import flops
    world, rank, local = init_ranks(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, k, v, _, offs = make_inputs(w, with_dout=False)
    pairs = flops.allowed_pairs(w.mask_kind, w.Nq, w.Nkv, w.window, offs)
    f_fwd = flops.attention_flops(w.B, w.Hq, w.d, pairs, backward=False)
    host = [t.pin_memory() for t in (q, k, v)]
    qd, kd, vd = (t.to(dev) for t in host)
    dt = None if offs is None else torch.from_numpy(np.asarray(offs, dtype=np.int32)).to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:-1], dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kw = dict(scale=w.scale, mask_kind=w.mask_kind, window=w.window, doc_offsets=dt,
              score_kind=w.score_kind, softcap=w.softcap)
    if fp8:
        (q8, sq), (k8, sk), (v8t, sv) = ea.fp8_inputs(qd, kd, vd)

        def fwd():
            ea.fwd_fp8_into(q8, sq, k8, sk, v8t, sv, o, lse, Nkv=w.Nkv, **kw)
    else:
        def fwd():
            ea.fwd_into(qd, kd, vd, o, lse, **kw)
    for _ in range(args.warmup):
        fwd()
    torch.cuda.synchronize()
    if ea.device_status() != 0:
        raise RuntimeError("a kernel gave up a bounded wait during warm-up")
    def timed_rep():
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for s in range(args.steps):
            flush.zero_()
            ev[s][0].record(stream)
            fwd()
            ev[s][1].record(stream)
        torch.cuda.synchronize()
        return [[e[0].elapsed_time(e[1])] for e in ev]

    rows, reps, clocks = repeat_timed(args, world, dev, timed_rep)
    if ea.device_status() != 0:
        raise RuntimeError("a kernel gave up a bounded wait during the timed steps")
    times = [r[0] for r in rows]
    t_all = sum(times)
    if world > 1:
        t_all = max_over_ranks(t_all, dev)
    ms_step = t_all / len(times)
    value = world * f_fwd / (ms_step * 1e-3) / 1e12
    outs_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in outs_host)
    in_sets = [(qd, kd, vd), tuple(torch.empty_like(t) for t in (qd, kd, vd))]
    out_sets = [(o, lse), (torch.empty_like(o), torch.empty_like(lse))]

    def run_step(x):  # the public call on buffer set x (FP8: quantise, then the FP8 forward)
        (bq, bk, bv), (bo, blse) = in_sets[x], out_sets[x]
        if fp8:
            (a8, a_s), (b8, b_s), (c8, c_s) = ea.fp8_inputs(bq, bk, bv)
            ea.fwd_fp8_into(a8, a_s, b8, b_s, c8, c_s, bo, blse, Nkv=w.Nkv, **kw)
        else:
            ea.fwd_into(bq, bk, bv, bo, blse, **kw)

    if world > 1:
        torch.distributed.barrier()
    ms_e2e = pipelined_e2e(args.steps, stream, dev, host, in_sets, out_sets, outs_host, run_step)
    pk = peaks()
    ach = f_fwd / (statistics.mean(times) * 1e-3) / 1e12
    tpeak, tpeak_name = tensor_peak(pk, sum(times))
    peak = tpeak * (2 if fp8 else 1)  # FP8 dense rate: 2x bf16 (nominal ratio)
    burst = pk["bf16_tflops"] * (2 if fp8 else 1)
    kname = "fwd256_kernel" if w.d == 256 else "fwd_tc_kernel"
    line = {
        "metric": ("attention FP8 forward TFLOP/s (unmasked FLOPs) and % of GB300 dense FP8 peak"
                   if fp8 else
                   "attention forward TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 peak"),
        "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic (seeded randn rounded to bf16" + (", quantised to e4m3)" if fp8 else ")"),
        "config": workload_config(w, {"parallelism": f"replicas x{world}",
                                      "pairs_per_head": pairs}),
        "pct_of_peak": round(100 * value / world / burst, 1),
        "kernels": {kname: {"ms": round(statistics.mean(times), 4),
                                      "min_ms": round(min(times), 4),
                                      "achieved": round(ach, 2), "unit": UNIT,
                                      "frac": round(ach / peak, 4)}},
        "roofline": {"bound": "tensor", "kernel": kname, "achieved": round(ach, 2),
                     "peak": peak, "unit": UNIT, "frac": round(ach / peak, 4),
                     "frac_of_burst": round(ach / burst, 4),
                     "peak_source": pk["source"] + " " + tpeak_name + (
                         " x 2 (nominal fp8/bf16 ratio)" if fp8 else ""),
                     "traffic": None},
        "e2e": {"value": round(world * f_fwd / (ms_e2e * 1e-3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 4)},
        "timed_repeats": reps, "timed_steps": len(times),
        "gpu_launches": len(times),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_forward(w, offs, seconds=args.cpu_seconds)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_decode(args, w):
    """Paged decode: a step is one attn_decode_paged call (the decode kernel and, when the
    keys are split, the combine kernel) over every sequence of the workload. The KV cache
    is resident state (uploaded once, like weights); a step's inputs are the new queries,
    the page table and the lengths."""
    from exact_io_aware_13_gb300 import build as libbuild
    libbuild.build()
    import exact_io_aware_13_gb300 as ea
    world, rank, local = init_ranks(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    q, kc, vc, table, lens = make_decode_inputs(w)
    host = [t.pin_memory() for t in (q, table, lens)]
    qd, td, ld = (t.to(dev) for t in host)
    kcd, vcd = kc.to(dev), vc.to(dev)
    del kc, vc
    total = int(lens.sum())
    kv_bytes = total * w.Hkv * w.d * 2 * 2
    io_bytes = kv_bytes + q.numel() * 2 * 2 + q.numel() // w.d * 4  # + Q in, O out, LSE out
    pairs = total * w.Hq * w.Nq  # every query sees every cached key (one decode token)
    f_step = 4 * w.d * pairs
    split = ea.decode_split_keys(w.B, w.Hq, w.Hkv, w.Nq, total)
    msl = w.len_max
    o = torch.empty((w.B, w.Hq, w.Nq, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    nws = ea.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.d, msl, split)
    ws = torch.empty((max(nws, 256),), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    kw = dict(max_seq_len=msl, split_keys=split, scale=w.scale, mask_kind=w.mask_kind,
              window=w.window, score_kind=w.score_kind, softcap=w.softcap)

    def step():
        ea.decode_paged_into(qd, kcd, vcd, td, ld, o, lse, ws if nws else None, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if ea.device_status() != 0:
        raise RuntimeError("a kernel reported a device error during warm-up")
    def timed_rep():
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
              for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        for s in range(args.steps):
            flush.zero_()
            ev[s][0].record(stream)
            step()
            ev[s][1].record(stream)
        torch.cuda.synchronize()
        return [[e[0].elapsed_time(e[1])] for e in ev]

    rows, reps, clocks = repeat_timed(args, world, dev, timed_rep)
    if ea.device_status() != 0:
        raise RuntimeError("a kernel reported a device error during the timed steps")
    times = [r[0] for r in rows]
    t_all = sum(times)
    if world > 1:
        t_all = max_over_ranks(t_all, dev)
    ms_step = t_all / len(times)
    gbs = world * io_bytes / (ms_step * 1e-3) / 1e9
    outs_host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in outs_host)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        for dst, src in zip((qd, td, ld), host):
            dst.copy_(src, non_blocking=True)
        step()
        for dst, src in zip(outs_host, (o, lse)):
            dst.copy_(src, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / args.steps
    pk = peaks()
    ms_mean = statistics.mean(times)
    ach = io_bytes / (ms_mean * 1e-3) / 1e9
    launches = 1 if nws == 0 else 2
    line = {
        "metric": "attention paged decode: GB/s of KV cache, queries and outputs moved, and % "
                  "of measured GB300 HBM copy bandwidth",
        "value": round(gbs, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded randn rounded to bf16; seeded lengths and shuffled pages)",
        "config": {"workload": w.describe(), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq,
                   "d": w.d, "page_size": w.page_size, "kv_tokens": total,
                   "split_keys": split, "seed": w.seed,
                   "parallelism": f"replicas x{world}",
                   "l2": f"flushed between steps (256 MiB write); KV cache {kv_bytes >> 20} MiB"},
        "pct_of_peak": round(100 * gbs / world / pk["hbm_gbs"], 1),
        "tflops": round(world * f_step / (ms_step * 1e-3) / 1e12, 2),
        "kernels": {"decode_tc_kernel+decode_combine_kernel": {
            "ms": round(ms_mean, 4), "min_ms": round(min(times), 4), "achieved": round(ach, 1),
            "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4)}},
        "roofline": {"bound": "hbm", "kernel": "decode_tc_kernel (+ combine, timed together)",
                     "achieved": round(ach, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(ach / pk["hbm_gbs"], 4),
                     "peak_source": pk["source"] + " HBM copy",
                     "traffic": ncu_traffic("decode_tc_kernel")},
        "e2e": {"value": round(world * io_bytes / (ms_e2e * 1e-3) / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(ms_e2e, 4)},
        "timed_repeats": reps, "timed_steps": len(times),
        "gpu_launches": launches * len(times),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(w, seconds=args.cpu_seconds)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def cpu_baseline(w, seconds: float = 20.0, heads: int = 1):
    """Time the float64 oracle (forward + backward) on `heads` (b, h) heads of the
    workload, full sequence, on the host cores."""
    import oracle
    from exact_io_aware_13_gb300 import flops
    q, k, v, do, _ = make_inputs(w)
    done, t0 = 0, time.perf_counter()
    pairs = flops.allowed_pairs(w.mask_kind, w.Nq, w.Nkv)
    while done < heads or (time.perf_counter() - t0 < seconds and done < w.B * w.Hq):
        b, h = divmod(done, w.Hq)
        sl = (slice(b, b + 1), slice(h, h + 1))
        drop = dict(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed)
        oracle.forward(q[sl], k[sl], v[sl], w.scale, mask_kind=w.mask_kind, **drop)
        oracle.backward(q[sl], k[sl], v[sl], do[sl], w.scale, mask_kind=w.mask_kind, **drop)
        done += 1
        if time.perf_counter() - t0 > seconds:
            break
    el = time.perf_counter() - t0
    f = flops.attention_flops(1, done, w.d, pairs, True) + flops.attention_flops(1, done, w.d,
                                                                                  pairs, False)
    return {"value": round(f / el / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(el, 6),
            "sample": f"{done} of {w.B * w.Hq} heads (full N={w.Nq}), forward + backward, "
                      "float64 numpy oracle (BLAS threads = all cores)"}


def cpu_baseline_forward(w, offs, seconds: float = 20.0, block: int = 512):
    """Time the float64 oracle's forward on blocks of `block` query rows of the workload's
    heads, taken in a seeded random order, on the host cores, for about `seconds` (at least
    one block). The value is the useful TFLOP/s of the rows done (allowed pairs only), the
    metric of the GPU line. The inputs are widened to float64 once, before the clock."""
    import oracle
    from exact_io_aware_13_gb300 import flops
    q, k, v, _, _ = make_inputs(w, with_dout=False)
    q64, k64, v64 = (t.to(torch.float64).numpy() for t in (q, k, v))
    n_blocks = -(-w.Nq // block)
    order = np.random.default_rng(0).permutation(w.B * w.Hq * n_blocks)
    done = []
    t0 = time.perf_counter()
    for idx in order:
        bh, rb = divmod(int(idx), n_blocks)
        b, h = divmod(bh, w.Hq)
        rows = np.arange(rb * block, min(w.Nq, (rb + 1) * block))
        oracle.forward(q64, k64, v64, w.scale, mask_kind=w.mask_kind, window=w.window,
                       doc_offsets=offs, score_kind=w.score_kind, softcap=w.softcap,
                       rows=rows, heads=[(b, h)], dropout_p=w.dropout_p,
                       dropout_seed=w.dropout_seed)
        done.append(rows)
        if time.perf_counter() - t0 > seconds:
            break
    el = time.perf_counter() - t0
    pairs = sum(flops.allowed_pairs_rows(w.mask_kind, r, w.Nkv, w.window, offs) for r in done)
    f = flops.attention_flops(1, 1, w.d, pairs, backward=False)
    n_rows = sum(len(r) for r in done)
    return {"value": round(f / el / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(el, 6),
            "sample": f"{len(done)} blocks of up to {block} query rows ({n_rows} of "
                      f"{w.B * w.Hq * w.Nq} rows, seeded order over heads), forward only, "
                      "float64 numpy oracle (BLAS threads = all cores)"}


def cpu_baseline_decode(w, seconds: float = 20.0):
    """Time the float64 decode oracle on (sequence, kv head) units of the decode workload,
    each with the G query heads that share its cache, in a seeded order, for about
    `seconds` (at least one unit). The value is GB/s of the bytes the GPU line counts for
    those units (their K and V once, Q in, O and LSE out). The caches are widened to
    float64 once, before the clock."""
    from oracle import decode_oracle
    q, kc, vc, table, lens = make_decode_inputs(w)
    q64 = q.to(torch.float64).numpy()
    kc64, vc64 = kc.to(torch.float64).numpy(), vc.to(torch.float64).numpy()
    G = w.Hq // w.Hkv
    order = np.random.default_rng(0).permutation(w.B * w.Hkv)
    nbytes, units = 0, 0
    t0 = time.perf_counter()
    for idx in order:
        b, g = divmod(int(idx), w.Hkv)
        decode_oracle.decode_forward(q64[b:b + 1], kc64, vc64, table[b:b + 1], lens[b:b + 1],
                                     w.scale, w.mask_kind, w.window, w.score_kind, w.softcap,
                                     heads=[(0, h) for h in range(g * G, (g + 1) * G)])
        nbytes += int(lens[b]) * w.d * 2 * 2 + G * w.Nq * (w.d * 2 * 2 + 4)
        units += 1
        if time.perf_counter() - t0 > seconds:
            break
    el = time.perf_counter() - t0
    return {"value": round(nbytes / el / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(),
            "kind": "oracle", "seconds": round(el, 6),
            "sample": f"{units} of {w.B * w.Hkv} (sequence, kv head) units with their {G} query "
                      "heads, float64 numpy decode oracle (BLAS threads = all cores)"}


REFERENCE_WORKLOADS = {"fwd_bwd": CAUSAL_FWD_BWD, "fwd_bwd_dropout": CAUSAL_FWD_BWD_DROPOUT,
                       "fwd_bwd_d256": CAUSAL_D256_FWD_BWD}


def run_reference(args):
    """The reference arm: the float64 oracle on the host cores, each step one bounded
    sample of the same workload (fwd+bwd: one head, forward and backward; forward-only:
    one block of query rows; decode: one (sequence, kv head) unit), with the metric and
    unit of our line. Only rank 0 runs; the other ranks exit without work."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    wl = args.workload
    if wl == "paged_decode":
        w = PAGED_DECODE
        samples = [cpu_baseline_decode(w, seconds=0.0) for _ in range(args.steps)]
        metric = ("attention paged decode: GB/s of KV cache, queries and outputs moved, and % "
                  "of measured GB300 HBM copy bandwidth")
        cfg = {"workload": w.describe(), "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq,
               "d": w.d, "page_size": w.page_size, "seed": w.seed}
        dtype = "f64"
    elif wl in FWD_WORKLOADS:
        w = FWD_WORKLOADS[wl]
        _, _, _, _, offs = make_inputs(w, with_dout=False)
        samples = [cpu_baseline_forward(w, offs, seconds=0.0) for _ in range(args.steps)]
        metric = "attention forward TFLOP/s (unmasked FLOPs) and % of GB300 dense BF16 peak"
        if wl.startswith("fp8"):
            metric = "attention FP8 forward TFLOP/s (unmasked FLOPs) and % of GB300 dense FP8 peak"
        cfg = workload_config(w)
        dtype = "f64"
    else:
        w = REFERENCE_WORKLOADS.get(wl, CAUSAL_FWD_BWD)
        samples = [cpu_baseline(w, seconds=0.0, heads=1) for _ in range(args.steps)]
        metric = METRIC
        cfg = workload_config(w)
        dtype = "f64"
    # every sample is one step: the line's value is total work over total time
    secs = [c["seconds"] for c in samples]
    value = sum(c["value"] * c["seconds"] for c in samples) / max(sum(secs), 1e-9)
    unit = samples[0]["unit"]
    ms = statistics.mean(secs) * 1e3
    cfg["sample"] = samples[0]["sample"] + " per step"
    line = {"impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded randn rounded to bf16)", "config": cfg,
            "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": cfg["sample"]},
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_cpu_replica_check(args):
    """The replica launcher and the cross-rank reduction on CPU: gloo ranks, each timing
    args.steps float64 256 x 256 matmuls; the job time is the maximum over ranks and the
    value sums the ranks' work over it, as in the GPU lines."""
    world, rank, _ = init_ranks(args, backend="gloo")
    a = np.random.default_rng(rank).standard_normal((256, 256))
    for _ in range(args.warmup):
        a @ a
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        a @ a
    ms = (time.perf_counter() - t0) * 1e3
    ms_rank = ms
    if world > 1:
        ms = max_over_ranks(ms, "cpu")
    work = 2.0 * 256 ** 3 * args.steps
    line = {"metric": "cpu replica check: GFLOP/s of float64 256x256 matmuls",
            "value": round(world * work / (ms * 1e-3) / 1e9, 4), "unit": "GFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms / args.steps, 6), "higher_is_better": True,
            "scaling": "weak", "rank0_ms": round(ms_rank, 6),
            "config": {"workload": "cpu replica check", "parallelism": f"replicas x{world}"}}
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--min-seconds", type=float, default=2.0)
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="fwd_bwd",
                    choices=["fwd_bwd", "fwd_bwd_dropout", "fwd_bwd_d256", *FWD_WORKLOADS,
                             "paged_decode", "cpu_replica_check"])
    args = ap.parse_args()
    if args.gpus < 1 or args.steps < 1:
        raise SystemExit("bench.py: --gpus and --steps must be at least 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        raise SystemExit(launch_replicas(args.gpus, sys.argv[1:]))
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "cpu_replica_check":
        run_cpu_replica_check(args)
    elif args.workload == "paged_decode":
        run_decode(args, PAGED_DECODE)
    elif args.workload == "fwd_bwd_dropout":
        run_ours(args, CAUSAL_FWD_BWD_DROPOUT)
    elif args.workload == "fwd_bwd_d256":
        run_ours(args, CAUSAL_D256_FWD_BWD)
    elif args.workload != "fwd_bwd":
        run_forward(args, FWD_WORKLOADS[args.workload], fp8=args.workload.startswith("fp8"))
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
