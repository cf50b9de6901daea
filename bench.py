#!/usr/bin/env python3
"""Benchmark: attention forward TFLOP/s on one GB300 (and % of dense tensor peak).

One step = one pass of the whole hot path over one batch: the tiled online-
softmax attention forward on the workload, non-causal then causal (the two
variants the base configuration names), FLOPs = 4*B*H*N^2*d each, halved for
causal.  Default workload: B=4, H=32, N=2048, d=64, fp16, scale 1/sqrt(64),
seeded iid N(0,1) inputs ("base").

Prints ONE JSON line (rank 0).  Keys beyond the metric: roofline (dominant
kernel = the non-causal launch), cpu_baseline (the fp64 oracle on host cores,
bounded row sample), e2e (pinned host buffers, H2D + compute + D2H per step),
clocks (nvidia-smi sampled during warm-up + timed region), gpu_launches.

--impl reference times the fp64 CPU oracle (the reference arm of this build)
on a bounded row sample of the same workload, on the host cores.

--op decode measures decoding attention (fa_decode: Nq <= 16 query rows per
head against a long KV sequence, split-KV) on a decoding workload
(--workload decode or decode_spec); it is HBM-bound, so its metric and
roofline are the bytes of K and V streamed per second against the measured
HBM bandwidth.

--op bwd measures the backward pass instead (fa_bwd: gradients of Q, K, V from
the forward's O and LSE and an upstream gradient dO), FLOPs = 2.5x the
forward's (five N x N x d products per head instead of two); its CPU legs time
the fp64 oracle's backward on a bounded sample of heads.

Multi-GPU (torchrun): each rank runs its own copy of the workload on its own
GPU (weak scaling; attention over (batch*head, Q tile) needs no exchange);
time = max over ranks; value = all ranks' FLOPs / that time.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s at 1 GB300 and % of dense FP16/BF16 tensor peak"
METRIC_BWD = "attention bwd TFLOP/s at 1 GB300 and % of dense FP16/BF16 tensor peak"
METRIC_DEC = "decoding attention K/V GB/s at 1 GB300 and % of measured HBM bandwidth"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
EX2_PER_CLOCK_PER_SM = 31.3  # measured ex2.approx.ftz.f32 rate (see the exp diagnostic below)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="base")
    ap.add_argument("--op", choices=["fwd", "bwd", "decode"], default="fwd",
                    help="fwd: the attention forward (the default step); bwd: the backward pass; "
                         "decode: decoding attention (use --workload decode / decode_spec)")
    ap.add_argument("--kernel", choices=["fa2", "fa1"], default="fa2",
                    help="fa2: the tiled FA2 forward (the product); fa1: the FA1-structured "
                         "baseline the pages compare it against")
    ap.add_argument("--variants", default="noncausal,causal",
                    help="comma list of noncausal/causal launches per step")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target host seconds for the cpu_baseline / reference sample")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="target total host seconds of the --impl reference run")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the d=128 and long-context target workloads in the forward line")
    ap.add_argument("--no-fa1-ratio", action="store_true",
                    help="skip the FA2 / FA1 timing table in the forward line")
    ap.add_argument("--target-steps", type=int, default=5,
                    help="timed steps per variant of each target workload")
    return ap.parse_args()


def flops_of(meta, causal):
    f = 4.0 * meta["B"] * meta["H"] * meta["N"] ** 2 * meta["d"]
    return f / 2 if causal else f


def bwd_flops_of(meta, causal):
    return 2.5 * flops_of(meta, causal)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# Sources each kernel's translation unit compiles: a recorded DRAM figure
# stays valid while these hash to the recorded value.
KERNEL_SOURCES = {
    "fa2": ("fa_fwd.cu", "fa_fwd_kernel.cuh", "fa1_fwd_kernel.cuh", "fa_common.cuh", "fa_host.h",
            "sm100_ptx.cuh"),
    "fa1": ("fa_fwd.cu", "fa_fwd_kernel.cuh", "fa1_fwd_kernel.cuh", "fa_common.cuh", "fa_host.h",
            "sm100_ptx.cuh"),
    "bwd": ("fa_bwd.cu", "fa_bwd_kernel.cuh", "fa_common.cuh", "fa_host.h", "sm100_ptx.cuh"),
    "decode": ("fa_decode.cu", "fa_decode_kernel.cuh", "fa_decode_tc_kernel.cuh", "fa_common.cuh", "fa_host.h",
               "sm100_ptx.cuh"),
}


def kernel_source_hash(kernel="fa2"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_02_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()


def recorded_traffic(workload, src_hash, kernel="fa2"):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, valid only while the kernel sources are the ones profiled."""
    stem = {"fa2": "fa_fwd", "fa1": "fa1_fwd", "bwd": "fa_bwd", "decode": "fa_decode"}[kernel]
    path = os.path.join(ROOT, "profiles", "%s_%s_dram.md" % (stem, workload))
    try:
        text = open(path).read()
    except OSError:
        return None, None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != src_hash:
        return None, path
    return float(m_bytes.group(1)), path


# ---------------------------------------------------------------------------
# clocks


class ClockSampler:
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = (uuid or "").lower()
        self.proc = None
        self.lines = []
        self.t_load = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark_load(self, t0, t1):
        self.t_load = (t0, t1)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summary(*(self.t_load or (0, float("inf"))))

    def summary(self, t0, t1):
        """Median SM clock, max clock / power and the throttle reasons seen
        in the samples taken between wall-clock times t0 and t1."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1].lower():
                continue
            if not (t0 <= ts <= t1):
                continue
            try:
                sm.append(float(parts[2]))
                smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for n, val in zip(names, parts[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed helpers


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(dist, value, device=None):
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(dist, value, device=None):
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)


def oracle_sample_rows(meta, n_rows, seed=12345):
    import numpy as np
    B, H, N = meta["B"], meta["H"], meta["N"]
    rng = np.random.default_rng(seed)
    flat = rng.choice(B * H * N, size=min(n_rows, B * H * N), replace=False)
    return np.stack([flat // N, flat % N], axis=1).astype(np.int64)


def oracle_row_flops(meta, rows, causal):
    import numpy as np
    if causal:
        return float(np.sum(4.0 * (rows[:, 1] + 1) * meta["d"]))
    return 4.0 * len(rows) * meta["N"] * meta["d"]


class OracleTimer:
    """Times the fp64 oracle (as it stands) on row samples of the workload."""

    def __init__(self, q, k, v, meta, variants):
        import oracle
        self.orc = oracle.get()
        self.meta = meta
        self.variants = variants
        self.q64 = q.double().numpy()
        self.k64 = k.double().numpy()
        self.v64 = v.double().numpy()
        self.threads = self.orc.default_threads()
        self.scale = meta["d"] ** -0.5

    def run(self, rows):
        t0 = time.perf_counter()
        flops = 0.0
        for causal in self.variants:
            self.orc.attention_rows(self.q64, self.k64, self.v64, rows, self.scale, causal=causal,
                                    threads=self.threads)
            flops += oracle_row_flops(self.meta, rows, causal)
        return time.perf_counter() - t0, flops

    def rows_for_seconds(self, seconds):
        """Calibrate: rows whose oracle time is about `seconds` (at most all rows)."""
        total = self.meta["B"] * self.meta["H"] * self.meta["N"]
        n = min(total, 64 * self.threads)
        while True:
            dt, _ = self.run(oracle_sample_rows(self.meta, n, seed=1))
            if dt >= 0.25 or n >= total:
                break
            n = min(total, n * 4)
        per_row = max(dt / n, 1e-9)
        return max(1, min(total, int(seconds / per_row)))


def oracle_full_flops(meta, variants):
    """The oracle's own fp64 work for every row of the workload (causal row i sees i + 1 keys)."""
    B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
    return sum((2.0 * B * H * N * (N + 1) * d) if c else (4.0 * B * H * N * N * d) for c in variants)


def cpu_baseline_obj(timer, seconds, seed=99):
    n = timer.rows_for_seconds(seconds)
    rows = oracle_sample_rows(timer.meta, n, seed=seed)
    dt, flops = timer.run(rows)
    rate = flops / dt
    return {"value": rate / 1e12, "unit": "TFLOP/s", "cores": timer.threads, "kind": "oracle",
            "rows_per_s": len(rows) * len(timer.variants) / dt,
            # not measured: the whole workload's oracle work at the sample's rate
            "extrapolated_full_s": oracle_full_flops(timer.meta, timer.variants) / rate,
            "sample": "%d random query rows of workload %s (of %d), variants %s, fp64 C oracle, "
                      "%.1f s" % (len(rows), timer.meta["name"],
                                   timer.meta["B"] * timer.meta["H"] * timer.meta["N"],
                                   "+".join("causal" if c else "noncausal" for c in timer.variants),
                                   dt)}


class OracleBwdTimer:
    """Times the fp64 oracle's backward (as it stands) on whole heads of the workload."""

    def __init__(self, q, k, v, do, meta, variants):
        import oracle
        self.orc = oracle.get()
        self.meta = meta
        self.variants = variants
        B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
        self.q64, self.k64, self.v64, self.do64 = (t.double().numpy().reshape(B * H, 1, N, d)
                                                   for t in (q, k, v, do))
        self.threads = self.orc.default_threads()
        self.scale = d ** -0.5

    def run(self, heads):
        """heads: head indices; each variant runs them as one batch over the threads."""
        import numpy as np
        sel = np.asarray(heads, dtype=np.int64)
        q, k, v, g = (x[sel].reshape(1, len(sel), self.meta["N"], self.meta["d"])
                      for x in (self.q64, self.k64, self.v64, self.do64))
        t0 = time.perf_counter()
        flops = 0.0
        one = dict(self.meta, B=1, H=len(sel))
        for causal in self.variants:
            self.orc.attention_bwd(q, k, v, g, self.scale, causal=causal, threads=self.threads)
            flops += bwd_flops_of(one, causal)
        return time.perf_counter() - t0, flops

    def threads_used(self, n_heads):
        """Threads the oracle starts for n_heads (it gives each ceil(n/threads) heads)."""
        per = -(-n_heads // min(self.threads, n_heads))
        return -(-n_heads // per)

    def heads_for_seconds(self, seconds):
        total = self.meta["B"] * self.meta["H"]
        n = min(total, self.threads)
        dt, _ = self.run(list(range(n)))
        per = max(dt / n, 1e-9)
        # whole rounds of `threads` heads (the oracle splits heads over threads)
        want = max(1, int(seconds / per))
        return max(1, min(total, want))


def cpu_baseline_bwd_obj(timer, seconds):
    n = timer.heads_for_seconds(seconds)
    heads = list(range(n))
    dt, flops = timer.run(heads)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": timer.threads_used(n),
            "kind": "oracle",
            "sample": "%d of %d heads of workload %s, variants %s, fp64 C oracle backward, %.1f s"
                      % (n, timer.meta["B"] * timer.meta["H"], timer.meta["name"],
                         "+".join("causal" if c else "noncausal" for c in timer.variants), dt)}


# ---------------------------------------------------------------------------


def main():
    args = parse_args()
    from attention_forward_02_gb300 import inputs

    world, rank, local = dist_env()
    if args.op == "decode":
        return run_decode_op(args, world, rank, local)
    variants = [v.strip() == "causal" for v in args.variants.split(",") if v.strip()]
    q, k, v, meta = inputs.make_workload(args.workload)
    meta["name"] = args.workload
    config = {"workload": "%s B=%d H=%d N=%d d=%d %s" % (args.workload, meta["B"], meta["H"],
                                                         meta["N"], meta["d"], meta["dtype"]),
              "B": meta["B"], "H": meta["H"], "N": meta["N"], "d": meta["d"],
              "scale": "1/sqrt(d)",
              "variants": ["causal" if c else "noncausal" for c in variants],
              "inputs": "seeded iid N(0,1), rounded to %s" % meta["dtype"],
              "l2": "flushed between timed steps (256 MiB write)",
              "parallelism": "dp%d (independent replicas)" % max(world, args.gpus)}
    step_flops = sum(flops_of(meta, c) for c in variants)
    config["kernel"] = args.kernel

    if args.op == "bwd":
        config["op"] = "backward (dQ, dK, dV from O, LSE and dO)"
        config["kernel"] = "fa_bwd"
        do = inputs.make_dout(meta["B"], meta["H"], meta["N"], meta["d"], meta["dtype"],
                              inputs.DOUT_SEEDS.get(args.workload, 3))
        config["inputs"] += "; dO seeded iid N(0,1) (seed %d)" % inputs.DOUT_SEEDS.get(args.workload, 3)
        if args.impl == "reference":
            return run_reference_bwd(args, q, k, v, do, meta, variants, config, world, rank)
        return run_bwd(args, q, k, v, do, meta, variants, config, world, rank, local)

    if args.impl == "reference":
        return run_reference(args, q, k, v, meta, variants, config, step_flops, world, rank)

    import torch
    import attention_forward_02_gb300 as fa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product has no CPU path)")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    fa.load()

    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    outs = [(torch.empty_like(qd), torch.empty((meta["B"], meta["H"], meta["N"]),
                                               dtype=torch.float32, device=dev)) for _ in variants]
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    scale = meta["d"] ** -0.5

    if args.kernel == "fa1":
        ws = torch.empty(fa.fa1_fwd_workspace_size(meta["B"], meta["H"], meta["N"], meta["d"]),
                         dtype=torch.uint8, device=dev)
        run = lambda q_, k_, v_, **kw: fa.fa1_fwd(q_, k_, v_, workspace=ws, **kw)
    else:
        run = fa.fa_fwd

    def step():
        for (o, lse), causal in zip(outs, variants):
            run(qd, kd, vd, o=o, lse=lse, scale=scale, causal=causal, stream=stream)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    t_load0 = time.time()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        step()
    torch.cuda.synchronize(dev)
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after warm-up: %s" % fa.fa_status_str(st))

    K = args.steps
    nv = len(variants)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nv + 1)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)  # let the host run ahead so launches queue back to back
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        for j, ((o, lse), causal) in enumerate(zip(outs, variants)):
            run(qd, kd, vd, o=o, lse=lse, scale=scale, causal=causal, stream=stream)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    t_load1 = time.time()
    sampler.mark_load(t_load0, t_load1)
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after timed region: %s" % fa.fa_status_str(st))

    step_ms = [ev[i][0].elapsed_time(ev[i][nv]) for i in range(K)]
    per_kernel_ms = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)] for j in range(nv)]
    total_ms = max_over_ranks(dist, sum(step_ms), dev)
    total_flops = sum_over_ranks(dist, step_flops * K, dev)
    value = total_flops / (total_ms / 1e3) / 1e12
    ms_per_step = total_ms / K

    # e2e through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(run, torch, q, k, v, meta, variants, dev, stream, scale, step_flops,
                      max(3, min(K, 50)), dist)

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    targets = None
    if not args.no_targets and args.kernel == "fa2":
        targets = time_targets(torch, fa, dev, stream, flush, peak, args.target_steps, sampler,
                               [w for w in ("d128", "long") if w != args.workload])
    fa1_ratio = None
    if not args.no_fa1_ratio and args.kernel == "fa2":
        fa1_ratio = time_fa2_vs_fa1(torch, fa, dev, stream, flush, args.target_steps)

    clocks = sampler.stop()
    dom = variants.index(False) if False in variants else 0  # the non-causal launch
    dom_causal = variants[dom]
    dom_ms = statistics.mean(per_kernel_ms[dom])
    achieved = flops_of(meta, dom_causal) / (dom_ms / 1e3) / 1e12
    src_hash = kernel_source_hash(args.kernel)
    traffic, traffic_src = recorded_traffic(args.workload, src_hash, args.kernel)
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": "%s_kernel<%d,%s,%s>" % ("fa_fwd" if args.kernel == "fa2" else "fa1_fwd",
                                                   meta["d"], "causal" if dom_causal else
                                                       "noncausal", meta["dtype"]),
                "peak_source": "%s bf16_tflops (burst; fp16 dense rate equals bf16)" % peak_src,
                "launch_ms": dom_ms,
                "algorithmic_flops_per_launch": flops_of(meta, dom_causal),
                "variants_tflops": {("causal" if c else "noncausal"):
                                    flops_of(meta, c) / (statistics.mean(per_kernel_ms[j]) / 1e3)
                                    / 1e12 for j, c in enumerate(variants)}}

    # Secondary limit at small head dims: one 2^x per score on the MUFU, against
    # 31.3 ex2.approx.ftz.f32 per clock per SM (a microbenchmark of 152 CTAs x
    # 512 threads on this GPU model; 38.6 when mixed 2:1 with the f32 -> f16x2
    # conversion) at the median SM clock of the timed region.
    exps = float(meta["B"] * meta["H"] * meta["N"] * meta["N"]) * (0.5 if dom_causal else 1.0)
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    ex2_peak = EX2_PER_CLOCK_PER_SM * sm_count * sm_mhz * 1e6
    roofline["exp_diagnostic"] = {"exps_per_launch": exps, "achieved_per_s": exps / (dom_ms / 1e3),
                                  "ex2_peak_per_s": ex2_peak, "frac": exps / (dom_ms / 1e3) / ex2_peak,
                                  "peak_source": "microbenchmark, %.1f per clock per SM x %d SMs x %.0f MHz"
                                                 % (EX2_PER_CLOCK_PER_SM, sm_count, sm_mhz)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        timer = OracleTimer(q, k, v, meta, variants)
        cpu = cpu_baseline_obj(timer, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "pct_of_peak": 100.0 * value / peak,
                "dtype": meta["dtype"], "data": "synthetic", "config": config,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": K * nv * 1, "wall_s_timed": t_wall}
        if targets is not None:
            line["targets"] = targets
        if fa1_ratio is not None:
            line["fa2_vs_fa1"] = fa1_ratio
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def time_launches(torch, run_one, stream, flush, steps, warmup=3, min_seconds=0.0):
    """Mean device time (ms) of run_one() over `steps` launches (more, up to
    400, if that many take under min_seconds of device time), each bracketed
    by CUDA events on the launching stream, with L2 flushed before every
    launch outside the timed bracket."""
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(warmup):
        flush.zero_()
        if i == warmup - 1:
            a0.record(stream)
        run_one()
        if i == warmup - 1:
            b0.record(stream)
    torch.cuda.synchronize()
    est_s = max(a0.elapsed_time(b0), 1e-3) / 1e3
    steps = max(steps, min(400, int(min_seconds / est_s) + 1))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        run_one()
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs), steps


def time_targets(torch, fa, dev, stream, flush, peak, steps, sampler, names):
    """The other workloads the >= 60 % target names (d=128 B=2 H=16 N=8192
    bf16 and the long context B=1 H=8 N=65536 d=128 fp16), both variants,
    timed like the headline: CUDA events per launch, L2 flushed between
    launches outside the events."""
    from attention_forward_02_gb300 import inputs
    out = {}
    for name in names:
        q, k, v, meta = inputs.make_workload(name)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        del q, k, v
        o = torch.empty_like(qd)
        lse = torch.empty((meta["B"], meta["H"], meta["N"]), dtype=torch.float32, device=dev)
        scale = meta["d"] ** -0.5
        t0 = time.time()
        res = {"config": "%s B=%d H=%d N=%d d=%d %s" % (name, meta["B"], meta["H"], meta["N"],
                                                         meta["d"], meta["dtype"])}
        for causal in (False, True):
            # at least ~0.3 s of launches per variant, so the clock sampler sees them
            ms, n = time_launches(torch, lambda: fa.fa_fwd(qd, kd, vd, o=o, lse=lse, scale=scale,
                                                           causal=causal, stream=stream),
                                  stream, flush, steps, min_seconds=0.3)
            tf = flops_of(meta, causal) / (ms / 1e3) / 1e12
            res["causal" if causal else "noncausal"] = {
                "tflops": tf, "frac": tf / peak, "launch_ms": ms, "steps": n,
                "algorithmic_flops_per_launch": flops_of(meta, causal)}
        st = fa.fa_last_device_status(stream.cuda_stream)
        if st != 0:
            raise SystemExit("device status after %s: %s" % (name, fa.fa_status_str(st)))
        res["clocks"] = sampler.summary(t0, time.time())
        res["peak"] = peak
        out[name] = res
        del qd, kd, vd, o, lse
        torch.cuda.empty_cache()
    return out


# The pages' FA2 / FA1 ratios on an RTX 5090, each kernel tuned, [4, 32, 2048, 64]
# fp16 ("Triton으로 FlashAttention 1·2 forward 구현하기", section "기준 shape").
PAGE_FA2_FA1 = {"noncausal": 2.16, "causal": 1.79}


def time_fa2_vs_fa1(torch, fa, dev, stream, flush, steps):
    """FA2 (fa_fwd) and the FA1-structured loop nest (fa1_fwd) timed in the
    same process on the page's shape [B, 32, 2048, 64] fp16, B in {1, 2, 4, 8},
    both variants; ratio = FA1 time / FA2 time."""
    from attention_forward_02_gb300 import inputs
    rows = []
    for B in (1, 2, 4, 8):
        q, k, v, meta = inputs.make_workload("sweep_b%d" % B)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        o = torch.empty_like(qd)
        lse = torch.empty((B, 32, 2048), dtype=torch.float32, device=dev)
        ws = torch.empty(fa.fa1_fwd_workspace_size(B, 32, 2048, 64), dtype=torch.uint8, device=dev)
        row = {"B": B}
        for causal in (False, True):
            t2, _ = time_launches(torch, lambda: fa.fa_fwd(qd, kd, vd, o=o, lse=lse, scale=0.125,
                                                           causal=causal, stream=stream),
                                  stream, flush, steps)
            t1, _ = time_launches(torch, lambda: fa.fa1_fwd(qd, kd, vd, o=o, lse=lse, scale=0.125,
                                                            causal=causal, workspace=ws,
                                                            stream=stream),
                                  stream, flush, steps)
            fl = flops_of(meta, causal)
            row["causal" if causal else "noncausal"] = {
                "fa2_ms": t2, "fa1_ms": t1, "ratio": t1 / t2,
                "fa2_tflops": fl / (t2 / 1e3) / 1e12, "fa1_tflops": fl / (t1 / 1e3) / 1e12}
        st = fa.fa_last_device_status(stream.cuda_stream)
        if st != 0:
            raise SystemExit("device status after the FA1 comparison: %s" % fa.fa_status_str(st))
        rows.append(row)
        del qd, kd, vd, o, lse, ws
        torch.cuda.empty_cache()
    return {"shape": "[B, 32, 2048, 64] fp16, scale 1/8", "ratio": "fa1_ms / fa2_ms",
            "rows": rows, "page_ratio_B4_rtx5090": PAGE_FA2_FA1}


def pipelined_e2e(torch, dev, steps, h2d, compute, d2h):
    """Runs `steps` end-to-end steps with the host->device copies of step i+1
    and the device->host copies of step i-1 overlapping the compute of step
    i: three streams, two device buffer sets, events for every dependency.
    h2d(b, stream), compute(b, stream), d2h(b, stream) enqueue one step's
    copies / kernels for buffer set b.  Every step moves all its bytes; the
    time runs from the first copy in to the last copy out.  Returns ms."""
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    start.record(s_in)
    for i in range(steps):
        b = i & 1
        if i >= 2:
            s_in.wait_event(comp_done[b])  # step i-2 has finished reading buffer set b
        h2d(b, s_in)
        in_done[b].record(s_in)
        s_comp.wait_event(in_done[b])
        if i >= 2:
            s_comp.wait_event(out_done[b])  # step i-2's results have been copied out
        compute(b, s_comp)
        comp_done[b].record(s_comp)
        s_out.wait_event(comp_done[b])
        d2h(b, s_out)
        out_done[b].record(s_out)
    end.record(s_out)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end)


def run_e2e(run, torch, q, k, v, meta, variants, dev, stream, scale, step_flops, steps, dist):
    """End to end through the public API from pinned host buffers: per step
    the H2D copy of q, k, v, every variant's launch, and the D2H copy of every
    variant's O and LSE.  Reported value: the pipelined run (copies of the
    neighbouring steps overlap this step's kernels); `serial` is the same
    steps one after another on one stream."""
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    B, H, N = meta["B"], meta["H"], meta["N"]
    houts = [(torch.empty_like(hq).pin_memory(), torch.empty((B, H, N), dtype=torch.float32).pin_memory())
             for _ in variants]
    dins = [tuple(torch.empty_like(hq, device=dev) for _ in range(3)) for _ in range(2)]
    douts = [[(torch.empty_like(hq, device=dev), torch.empty((B, H, N), dtype=torch.float32, device=dev))
              for _ in variants] for _ in range(2)]
    h2d = 3 * hq.numel() * hq.element_size()
    d2h = sum(o.numel() * o.element_size() + l.numel() * 4 for o, l in houts)

    def copy_in(b, st):
        with torch.cuda.stream(st):
            for dst, src in zip(dins[b], (hq, hk, hv)):
                dst.copy_(src, non_blocking=True)

    def compute(b, st):
        qd, kd, vd = dins[b]
        for (o, l), causal in zip(douts[b], variants):
            run(qd, kd, vd, o=o, lse=l, scale=scale, causal=causal, stream=st)

    def copy_out(b, st):
        with torch.cuda.stream(st):
            for (o, l), (ho, hl) in zip(douts[b], houts):
                ho.copy_(o, non_blocking=True)
                hl.copy_(l, non_blocking=True)

    def serial_step():
        copy_in(0, stream)
        compute(0, stream)
        copy_out(0, stream)

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_serial = e0.elapsed_time(e1)
    pipelined_e2e(torch, dev, 3, copy_in, compute, copy_out)  # warm-up of the streams
    if dist is not None:
        dist.barrier()
    ms = pipelined_e2e(torch, dev, steps, copy_in, compute, copy_out)
    flops = step_flops * steps
    if dist is not None:
        ms = max_over_ranks(dist, ms, dev)
        ms_serial = max_over_ranks(dist, ms_serial, dev)
        flops = sum_over_ranks(dist, flops, dev)
    return {"value": flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "mode": "pipelined: step i+1's H2D and step i-1's D2H overlap step i's kernels "
                    "(3 streams, 2 device buffer sets)",
            "serial": {"value": flops / (ms_serial / 1e3) / 1e12, "ms_per_step": ms_serial / steps}}


def run_reference(args, q, k, v, meta, variants, config, step_flops, world, rank):
    """The reference arm: the fp64 CPU oracle, as it stands, on host cores."""
    if rank != 0:
        return
    timer = OracleTimer(q, k, v, meta, variants)
    budget = max(0.5, args.ref_seconds)
    n_steps = args.steps + max(args.warmup, 0)
    rows_per_step = timer.rows_for_seconds(budget / max(n_steps, 1))
    for i in range(max(args.warmup, 0)):
        timer.run(oracle_sample_rows(meta, rows_per_step, seed=500 + i))
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = timer.run(oracle_sample_rows(meta, rows_per_step, seed=1000 + i))
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = ("each step: %d random query rows of %s (of %d), variants %s, fp64 C oracle"
              % (rows_per_step, args.workload, meta["B"] * meta["H"] * meta["N"],
                 "+".join(config["variants"])))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": timer.threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_bwd(args, q, k, v, do, meta, variants, config, world, rank, local):
    """The backward pass: one step = fa_bwd for each variant (inputs resident)."""
    import torch
    import attention_forward_02_gb300 as fa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product has no CPU path)")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    fa.load()
    B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
    scale = d ** -0.5
    stream = torch.cuda.current_stream(dev)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    fwd = [fa.fa_fwd(qd, kd, vd, scale=scale, causal=c) for c in variants]  # the backward's inputs
    grads = [tuple(torch.empty_like(qd) for _ in range(3)) for _ in variants]
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def run_one(j, causal):
        o, lse = fwd[j]
        dq, dk, dv = grads[j]
        fa.fa_bwd(qd, kd, vd, o, lse, dod, scale=scale, causal=causal, dq=dq, dk=dk, dv=dv,
                  workspace=ws, stream=stream)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    t_load0 = time.time()
    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        for j, c in enumerate(variants):
            run_one(j, c)
    torch.cuda.synchronize(dev)
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after warm-up: %s" % fa.fa_status_str(st))
    K = args.steps
    nv = len(variants)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nv + 1)] for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)
    for i in range(K):
        flush.zero_()
        ev[i][0].record(stream)
        for j, c in enumerate(variants):
            run_one(j, c)
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    sampler.mark_load(t_load0, time.time())
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after timed region: %s" % fa.fa_status_str(st))
    step_flops = sum(bwd_flops_of(meta, c) for c in variants)
    step_ms = [ev[i][0].elapsed_time(ev[i][nv]) for i in range(K)]
    per_call_ms = [[ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)] for j in range(nv)]
    total_ms = max_over_ranks(dist, sum(step_ms), dev)
    value = sum_over_ranks(dist, step_flops * K, dev) / (total_ms / 1e3) / 1e12

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e_bwd(fa, torch, q, k, v, do, meta, variants, dev, stream, scale, step_flops,
                          max(3, min(K, 20)), dist)
    clocks = sampler.stop()
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    dom = variants.index(False) if False in variants else 0
    dom_ms = statistics.mean(per_call_ms[dom])
    achieved = bwd_flops_of(meta, variants[dom]) / (dom_ms / 1e3) / 1e12
    traffic, _ = recorded_traffic(args.workload, kernel_source_hash("bwd"), "bwd")
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "kernel": "fa_bwd_kernel<%d,%s,%s>" % (d, "causal" if variants[dom] else "noncausal",
                                                       meta["dtype"]),
                "timed": "the whole fa_bwd call (row-term kernel + main kernel + dQ rounding); "
                         "the main kernel's own rate is higher by its share of the call",
                "peak_source": "%s bf16_tflops (burst; fp16 dense rate equals bf16)" % peak_src,
                "launch_ms": dom_ms,
                "algorithmic_flops_per_launch": bwd_flops_of(meta, variants[dom]),
                "variants_tflops": {("causal" if c else "noncausal"):
                                    bwd_flops_of(meta, c) / (statistics.mean(per_call_ms[j]) / 1e3)
                                    / 1e12 for j, c in enumerate(variants)}}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline_bwd_obj(OracleBwdTimer(q, k, v, do, meta, variants), args.cpu_seconds)
    if rank == 0:
        line = {"metric": METRIC_BWD, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "pct_of_peak": 100.0 * value / peak, "dtype": meta["dtype"], "data": "synthetic",
                "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "clocks": clocks, "gpu_launches": K * nv * 3, "wall_s_timed": t_wall}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e_bwd(fa, torch, q, k, v, do, meta, variants, dev, stream, scale, step_flops, steps, dist):
    """Backward through the public API from pinned host buffers: per step and
    variant the H2D copy of q, k, v, o, lse, dO (o, lse made once by the
    forward), the backward, and the D2H copy of dq, dk, dv.  Pipelined as the
    forward's e2e; `serial` is the same steps on one stream."""
    B, H, N, d = meta["B"], meta["H"], meta["N"], meta["d"]
    hq, hk, hv, hdo = (t.pin_memory() for t in (q, k, v, do))
    host_fwd = []
    for c in variants:
        o, l = fa.fa_fwd(hq.to(dev), hk.to(dev), hv.to(dev), scale=scale, causal=c)
        host_fwd.append((o.cpu().pin_memory(), l.cpu().pin_memory()))
    outs_h = [tuple(torch.empty_like(hq).pin_memory() for _ in range(3)) for _ in variants]
    # per buffer set and variant: q, k, v, dO, o (16-bit) + lse; grads; a workspace
    dins = [[(tuple(torch.empty_like(hq, device=dev) for _ in range(5)),
              torch.empty((B, H, N), dtype=torch.float32, device=dev)) for _ in variants] for _ in range(2)]
    dgrads = [[tuple(torch.empty_like(hq, device=dev) for _ in range(3)) for _ in variants] for _ in range(2)]
    wss = [torch.empty(fa.fa_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev) for _ in range(2)]
    h2d = len(variants) * (5 * hq.numel() * hq.element_size() + B * H * N * 4)
    d2h = len(variants) * 3 * hq.numel() * hq.element_size()

    def copy_in(b, st):
        with torch.cuda.stream(st):
            for ((t16, ld), (ho, hl)) in zip(dins[b], host_fwd):
                for dst, src in zip(t16, (hq, hk, hv, hdo, ho)):
                    dst.copy_(src, non_blocking=True)
                ld.copy_(hl, non_blocking=True)

    def compute(b, st):
        for ((qd, kd, vd, dod, od), ld), g, c in zip(dins[b], dgrads[b], variants):
            fa.fa_bwd(qd, kd, vd, od, ld, dod, scale=scale, causal=c, dq=g[0], dk=g[1], dv=g[2],
                      workspace=wss[b], stream=st)

    def copy_out(b, st):
        with torch.cuda.stream(st):
            for g, hg in zip(dgrads[b], outs_h):
                for src, dst in zip(g, hg):
                    dst.copy_(src, non_blocking=True)

    def serial_step():
        copy_in(0, stream)
        compute(0, stream)
        copy_out(0, stream)

    for _ in range(3):
        serial_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        serial_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms_serial = e0.elapsed_time(e1)
    pipelined_e2e(torch, dev, 3, copy_in, compute, copy_out)
    if dist is not None:
        dist.barrier()
    ms = pipelined_e2e(torch, dev, steps, copy_in, compute, copy_out)
    flops = step_flops * steps
    if dist is not None:
        ms = max_over_ranks(dist, ms, dev)
        ms_serial = max_over_ranks(dist, ms_serial, dev)
        flops = sum_over_ranks(dist, flops, dev)
    return {"value": flops / (ms / 1e3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": ms / steps,
            "mode": "pipelined: step i+1's H2D and step i-1's D2H overlap step i's kernels "
                    "(3 streams, 2 device buffer sets)",
            "serial": {"value": flops / (ms_serial / 1e3) / 1e12, "ms_per_step": ms_serial / steps}}


def run_reference_bwd(args, q, k, v, do, meta, variants, config, world, rank):
    """The reference arm for the backward: the fp64 oracle's backward on host cores."""
    if rank != 0:
        return
    timer = OracleBwdTimer(q, k, v, do, meta, variants)
    budget = max(0.5, args.ref_seconds)
    n_steps = args.steps + max(args.warmup, 0)
    heads = timer.heads_for_seconds(budget / max(n_steps, 1))
    total = meta["B"] * meta["H"]
    for i in range(max(args.warmup, 0)):
        timer.run([(i * heads + h) % total for h in range(heads)])
    tot_t, tot_f = 0.0, 0.0
    for i in range(args.steps):
        dt, fl = timer.run([((i + args.warmup) * heads + h) % total for h in range(heads)])
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = ("each step: %d of %d heads of %s, variants %s, fp64 C oracle backward"
              % (heads, total, args.workload, "+".join(config["variants"])))
    print(json.dumps({"impl": "reference", "metric": METRIC_BWD, "value": value, "unit": "TFLOP/s",
                      "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": config,
                      "cpu_baseline": {"value": value, "unit": "TFLOP/s",
                                       "cores": timer.threads_used(heads), "kind": "oracle",
                                       "sample": sample},
                      "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}), flush=True)


# ---------------------------------------------------------------------------
# decoding


DECODE_NO_FLUSH_BYTES = 1 << 30  # K/V above 1 GiB (8x L2) are timed without a flush


def decode_bytes(meta):
    """Algorithmic bytes of one decoding call: K and V once, Q in, O out (16-bit), LSE (fp32)."""
    BH, Nq, Nk, d = meta["B"] * meta["H"], meta["Nq"], meta["Nk"], meta["d"]
    return BH * (2 * Nk * d * 2 + 2 * Nq * d * 2 + Nq * 4)


def decode_flops(meta):
    BH, Nq, Nk, d = meta["B"] * meta["H"], meta["Nq"], meta["Nk"], meta["d"]
    if meta["causal"]:
        keys = sum(Nk - Nq + i + 1 for i in range(Nq))
        return 4.0 * BH * keys * d
    return 4.0 * BH * Nq * Nk * d


class OracleDecodeTimer:
    """Times the fp64 oracle's decoding definition (as it stands) on whole heads;
    the sampled heads are widened to fp64 per call (a KV cache in fp64 would
    not fit the host)."""

    def __init__(self, q, k, v, meta):
        import oracle
        self.orc = oracle.get()
        self.meta = meta
        B, H = meta["B"], meta["H"]
        self.q = q.reshape(B * H, meta["Nq"], meta["d"])
        self.k = k.reshape(B * H, meta["Nk"], meta["d"])
        self.v = v.reshape(B * H, meta["Nk"], meta["d"])
        self.threads = self.orc.default_threads()

    def run(self, heads):
        import torch
        sel = torch.as_tensor(list(heads), dtype=torch.long)
        n = len(sel)
        q64 = self.q[sel].double().numpy().reshape(1, n, self.meta["Nq"], self.meta["d"])
        k64 = self.k[sel].double().numpy().reshape(1, n, self.meta["Nk"], self.meta["d"])
        v64 = self.v[sel].double().numpy().reshape(1, n, self.meta["Nk"], self.meta["d"])
        t0 = time.perf_counter()
        self.orc.attention_decode(q64, k64, v64, self.meta["d"] ** -0.5, causal=self.meta["causal"],
                                  threads=self.threads)
        dt = time.perf_counter() - t0
        one = dict(self.meta, B=1, H=n)
        return dt, decode_bytes(one)

    def heads_for_seconds(self, seconds):
        total = self.meta["B"] * self.meta["H"]
        n = min(total, 4 * self.threads)
        dt, _ = self.run(list(range(n)))
        return max(1, min(total, int(seconds / max(dt / n, 1e-9))))

    def threads_used(self, n_rows):
        return min(self.threads, n_rows)


def run_decode_op(args, world, rank, local):
    from attention_forward_02_gb300 import inputs
    name = args.workload if args.workload in inputs.DECODE_WORKLOADS else "decode"
    q, k, v, meta = inputs.make_decode_workload(name)
    meta["name"] = name
    B, H, Nq, Nk, d = meta["B"], meta["H"], meta["Nq"], meta["Nk"], meta["d"]
    kv_bytes = 2 * B * H * Nk * d * 2
    config = {"workload": "%s B=%d H=%d Nq=%d Nk=%d d=%d %s %s" % (
                  name, B, H, Nq, Nk, d, meta["dtype"], "causal (queries at the end)" if meta["causal"]
                  else "non-causal"),
              "B": B, "H": H, "Nq": Nq, "Nk": Nk, "d": d, "scale": "1/sqrt(d)",
              "inputs": "seeded iid N(0,1), rounded to %s" % meta["dtype"],
              "l2": ("K/V (%.2f GB) exceed L2 (129 MB) many times over: no flush between timed steps"
                     % (kv_bytes / 1e9) if kv_bytes > DECODE_NO_FLUSH_BYTES else
                     "flushed between timed steps (256 MiB write)"),
              "parallelism": "dp%d (independent replicas)" % max(world, args.gpus),
              "op": "decoding attention (split-KV)", "kernel": "fa_decode"}
    step_bytes = decode_bytes(meta)
    if args.impl == "reference":
        if rank != 0:
            return
        timer = OracleDecodeTimer(q, k, v, meta)
        n_steps = args.steps + max(args.warmup, 0)
        heads = timer.heads_for_seconds(max(0.5, args.ref_seconds) / max(n_steps, 1))
        total = B * H
        for i in range(max(args.warmup, 0)):
            timer.run([(i * heads + h) % total for h in range(heads)])
        tot_t, tot_b = 0.0, 0.0
        for i in range(args.steps):
            dt, by = timer.run([((i + args.warmup) * heads + h) % total for h in range(heads)])
            tot_t += dt
            tot_b += by
        value = tot_b / tot_t / 1e9
        sample = "each step: %d of %d heads of %s, fp64 C oracle" % (heads, total, name)
        print(json.dumps({"impl": "reference", "metric": METRIC_DEC, "value": value, "unit": "GB/s",
                          "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                          "config": config,
                          "cpu_baseline": {"value": value, "unit": "GB/s",
                                           "cores": timer.threads_used(heads * Nq), "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return

    import torch
    import attention_forward_02_gb300 as fa
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product has no CPU path)")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dist = init_dist(world, "nccl")
    fa.load()
    scale = d ** -0.5
    stream = torch.cuda.current_stream(dev)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(B, H, Nq, Nk, d), dtype=torch.uint8, device=dev)
    # a K/V cache many times the size of L2 is its own flush: a write flush would
    # only add its dirty lines' write-back to the timed HBM traffic
    flush = (torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
             if kv_bytes <= DECODE_NO_FLUSH_BYTES else None)

    def call(qq, oo, ll):
        fa.fa_decode(qq, kd, vd, o=oo, lse=ll, scale=scale, causal=meta["causal"], workspace=ws,
                     stream=stream)

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    t_load0 = time.time()
    for _ in range(max(args.warmup, 3)):
        if flush is not None:
            flush.zero_()
        call(qd, o, lse)
    torch.cuda.synchronize(dev)
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after warm-up: %s" % fa.fa_status_str(st))
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.perf_counter()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev[i][0].record(stream)
        call(qd, o, lse)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall0
    sampler.mark_load(t_load0, time.time())
    st = fa.fa_last_device_status(stream.cuda_stream)
    if st != 0:
        raise SystemExit("device status after timed region: %s" % fa.fa_status_str(st))
    ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(dist, sum(ms), dev)
    value = sum_over_ranks(dist, step_bytes * K, dev) / (total_ms / 1e3) / 1e9

    # e2e: per step the new queries go host -> device and O, LSE come back;
    # the KV cache is device-resident state, as in a decoding loop
    e2e = None
    if not args.no_e2e:
        hq = q.pin_memory()
        ho = torch.empty_like(hq).pin_memory()
        hl = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
        qq = torch.empty_like(qd)
        steps_e = max(3, min(K, 50))

        def one():
            qq.copy_(hq, non_blocking=True)
            call(qq, o, lse)
            ho.copy_(o, non_blocking=True)
            hl.copy_(lse, non_blocking=True)

        for _ in range(3):
            one()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps_e):
            one()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ems = max_over_ranks(dist, e0.elapsed_time(e1), dev)
        e2e = {"value": sum_over_ranks(dist, step_bytes * steps_e, dev) / (ems / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": hq.numel() * hq.element_size(),
               "d2h_bytes_per_step": ho.numel() * ho.element_size() + hl.numel() * 4,
               "steps": steps_e, "ms_per_step": ems / steps_e,
               "note": "KV cache resident on the device (decoding state), queries in and O/LSE out per step"}
    clocks = sampler.stop()
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    launch_ms = statistics.mean(ms)
    achieved = step_bytes / (launch_ms / 1e3) / 1e9
    traffic, _ = recorded_traffic(name, kernel_source_hash("decode"), "decode")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic,
                "kernel": ("fa_decode_tc_kernel<%d,%s> + combine" % (d, meta["dtype"])
                           if Nq >= 3 or (Nq == 2 and d == 128) else
                           "fa_decode_split_kernel<%d,%s> + combine" % (d, meta["dtype"])),
                "timed": "the whole fa_decode call (split kernel + combine kernel)",
                "peak_source": "%s hbm_gbs (STREAM-style copy)" % peak_src,
                "launch_ms": launch_ms, "algorithmic_bytes_per_launch": step_bytes,
                "tflops": decode_flops(meta) / (launch_ms / 1e3) / 1e12}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        timer = OracleDecodeTimer(q, k, v, meta)
        n = timer.heads_for_seconds(args.cpu_seconds)
        dt, by = timer.run(list(range(n)))
        cpu = {"value": by / dt / 1e9, "unit": "GB/s", "cores": timer.threads_used(n * Nq), "kind": "oracle",
               "sample": "%d of %d heads of workload %s, fp64 C oracle, %.1f s" % (n, B * H, name, dt)}
    if rank == 0:
        print(json.dumps({"metric": METRIC_DEC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
                          "warmup": args.warmup, "ms_per_step": total_ms / K, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "pct_of_peak": 100.0 * value / peak,
                          "dtype": meta["dtype"], "data": "synthetic", "config": config,
                          "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                          "gpu_launches": 2 * K, "wall_s_timed": t_wall}), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
