#!/usr/bin/env python
"""Benchmark of the batched tree speculative-sampling verify step on GB300.

One step = one spec_verify_tree call (tree preparation, dense row pass, accept
walk) over one batch of synthetic, seeded trees whose logits are already resident
in HBM.  The headline workload is B=64 trees of 60 nodes over V=128256 bf16 logits
(T=0.7, top-p 0.9); its target and draft logits (1.97 GB) are larger than the L2,
so no flush is needed between steps.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead
(rank 0 only; other ranks exit 0).  Under torchrun each rank verifies its own
batch of trees (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_tree_spec_gb300 import workloads as wl  # noqa: E402

METRIC = "verified draft-node logit rows/sec and achieved HBM GB/s vs GB300 peak (1 GPU)"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "tree60_b64_v128256"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
REFERENCE_BUDGET_S = 90.0  # host seconds the reference arm's timed sample may take
ROW_PASS_SOURCES = ["speculative_decoding_tree_spec_gb300/csrc/rows.cu",
                    "speculative_decoding_tree_spec_gb300/csrc/select.cuh",
                    "speculative_decoding_tree_spec_gb300/csrc/common.cuh",
                    "speculative_decoding_tree_spec_gb300/csrc/internal.h"]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--seed", type=int, default=20261202)
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (small cases for profiling)")
    ap.add_argument("--e2e-steps", type=int, default=12)
    ap.add_argument("--cpu-trees", type=int, default=48,
                    help="tree-steps in the oracle sample of the cpu_baseline leg")
    ap.add_argument("--host-threads", type=int, default=0,
                    help="host threads of the oracle legs (reference arm, cpu_baseline); "
                         "0 = every core")
    ap.add_argument("--ref-seconds", type=float, default=REFERENCE_BUDGET_S,
                    help="host seconds the reference arm's timed sample may take")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["verify", "commit", "tree", "draft"], default="verify",
                    help="commit: time the accepted-path commit on a KV cache instead; tree: "
                         "the EAGLE-2 dynamic draft-tree build (expansion + rerank + mask); "
                         "draft: the draft-side top-k drafting of the expanded nodes' rows")
    ap.add_argument("--fused", action="store_true",
                    help="with --op draft: the draft LM head + top-k in one call (features x "
                         "weight on the tensor cores, then the ranking kernel)")
    ap.add_argument("--per-request", action="store_true",
                    help="per-request sampling parameters: the trees cycle through greedy, the "
                         "workload's own setting, top-k 50 at T=1 and top-p 0.8 at T=0.5 "
                         "(spec_verify_tree_per_request); reported as its own line")
    ap.add_argument("--visited-only", action="store_true",
                    help="the visited-rows-only schedule (no dense pass); reported as its own "
                         "line, not the dense schedule's number")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def shard_seed(seed: int, rank: int) -> int:
    """Each rank draws its own independent batch of trees."""
    return seed + 1000003 * rank


def whole_job_rate(world: int, units_per_step: int, steps: int, elapsed_ms_max: float) -> float:
    """Units per second over all ranks: every rank does units_per_step per step, and the
    job takes as long as its slowest rank."""
    return world * units_per_step * steps / (elapsed_ms_max / 1e3)


# ---------------------------------------------------------------------------
# peaks, clocks, profiles
# ---------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (libnvidia-ml, by ctypes)
    every `period_ms` in a background thread: fine enough to put several samples inside a
    timed region of a few milliseconds.  Only reads; changes no setting."""
    # clock-event reason bits of NVML's public API
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, period_ms: float = 1.0):
        import ctypes
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            self.dev = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.dev)) != 0:
                return
            self.lib = lib
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            self.sm_max = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(
                self.dev, 1, ctypes.byref(mx)) == 0 else None
        except (OSError, AttributeError, RuntimeError):
            return
        self.ok = True
        self.period = period_ms / 1e3
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        import ctypes
        sm, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.time()
            a = self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ctypes.byref(sm))
            b = self.lib.nvmlDeviceGetPowerUsage(self.dev, ctypes.byref(pw))
            c = self.reasons_fn(self.dev, ctypes.byref(rs))
            self.samples.append((t, sm.value if a == 0 else None, pw.value / 1e3 if b == 0 else None,
                                 rs.value if c == 0 else 0))
            time.sleep(self.period)

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.ok and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.001)

    def stop(self):
        self._stop.set()
        if self.ok:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [r for r in self.samples if t0 <= r[0] <= t1]
        sm = [r[1] for r in rows if r[1] is not None]
        reasons = set()
        for r in rows:
            for bit, name in self.REASONS.items():
                if r[3] & bit:
                    reasons.add(name)
        power = [r[2] for r in rows if r[2] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": self.sm_max,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None, "source": "nvml, 1 ms period"}


def clock_sampler(device_index: int):
    """NVML sampling where the library loads, else nvidia-smi."""
    s = NvmlClockSampler(device_index)
    return s if s.ok else ClockSampler(device_index)


class ClockSampler:
    """nvidia-smi sampling of SM clock, power and throttle reasons in a background thread."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index: int, period_ms: int = 50):
        self.samples = []
        self.proc = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid]
        except Exception:
            sel = []
        cmd = ["nvidia-smi", f"--query-gpu={','.join(self.FIELDS)}", "--format=csv,noheader,nounits",
               f"-lms={period_ms}"] + sel
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def wait_first(self, timeout=5.0):
        t0 = time.time()
        while self.proc is not None and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.02)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        rows = [s for t, s in self.samples if t0 <= t <= t1 and len(s) == len(self.FIELDS)]
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = set()
        for r in rows:
            for name, val in zip(["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                  "sw_power_cap"], r[3:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        power = [num(r[2]) for r in rows if num(r[2]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(power) if power else None}


WALK_SOURCES = ["speculative_decoding_tree_spec_gb300/csrc/walk.cu",
                "speculative_decoding_tree_spec_gb300/csrc/select.cuh",
                "speculative_decoding_tree_spec_gb300/csrc/common.cuh",
                "speculative_decoding_tree_spec_gb300/csrc/internal.h"]
DRAFT_SOURCES = ["speculative_decoding_tree_spec_gb300/csrc/draft.cu",
                 "speculative_decoding_tree_spec_gb300/csrc/common.cuh",
                 "speculative_decoding_tree_spec_gb300/csrc/internal.h"]


def sources_digest(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, profile: str = "row_pass", sources=None):
    """Per-launch DRAM traffic of a kernel from its committed ncu summary
    (profiles/<profile>_<workload>.md), if it was captured on the kernel's current
    sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{profile}_{workload}.md")
    if not os.path.exists(path):
        return None, None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not d:
        return None, None
    if d.group(1) != sources_digest(sources or ROW_PASS_SOURCES):
        return None, "stale"
    return float(m.group(1)), "current"


# ---------------------------------------------------------------------------
# the oracle leg (CPU baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_pool(w, seed, n_trees, device):
    """Host copies of n_trees trees of workload w (the oracle's input format)."""
    small = w.with_(B=n_trees)
    inp = wl.build_inputs(small, seed=seed, device=device)
    return {"p": wl.host_logits(inp["p"]), "q": wl.host_logits(inp["q"]),
            "tokens": inp["tokens"], "parents": inp["parents"], "max_depth": inp["max_depth"]}


def time_oracle(w, pool, n_steps, threads, seed):
    """n_steps tree-steps (step k verifies pool tree k mod P, drawing as batch index k)
    on `threads` host threads.  Returns (wall seconds, rows verified)."""
    import oracle

    P = pool["p"].shape[0]

    def step(k):
        j = k % P
        oracle.verify_tree(pool["p"][j:j + 1], pool["q"][j:j + 1], pool["tokens"][j:j + 1],
                           pool["parents"][j:j + 1], pool["max_depth"], w.temperature, w.top_k,
                           w.top_p, seed=seed, offset=0, batch_index=k)

    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(step, range(n_steps)))
    return time.perf_counter() - t0, n_steps * w.N


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle

    oracle.build()
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    threads = args.host_threads or os.cpu_count() or 1
    pool = oracle_pool(w, args.seed, min(16, w.B), "cpu")
    # a step is one tree verified by the oracle; the timed sample is bounded so that
    # the run ends within a few minutes whatever --steps asks for
    n_warm = max(1, min(args.warmup, threads))
    wall_w, _ = time_oracle(w, pool, n_warm, threads, args.seed)
    per_step = wall_w / n_warm
    # at least two tree-steps per host thread, so that every thread stays busy over the
    # sample; beyond that as many of the requested steps as the time budget allows
    n_timed = max(2 * threads, min(args.steps, int(args.ref_seconds / max(per_step, 1e-9))))
    wall, rows = time_oracle(w, pool, n_timed, threads, args.seed)
    value = rows / wall
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / n_timed,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "V": w.V, "logits": w.dtype,
                   "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p,
                   "step": "one tree verified by the CPU oracle (steps run on a host thread pool)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{n_timed} of the {args.steps} requested tree-steps timed "
                                   f"(at most {args.ref_seconds:.0f} s of host time), cycling "
                                   f"over {pool['p'].shape[0]} seeded trees of {w.name}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    from speculative_decoding_tree_spec_gb300 import binding

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    if w.logits == "lmhead":
        return run_ours_lmhead(args, w, world, rank, local, dev)
    seed = shard_seed(args.seed, rank)
    inp = wl.build_inputs(w, seed=seed, device=dev)
    tok = torch.as_tensor(inp["tokens"], device=dev)
    par = torch.as_tensor(inp["parents"], device=dev)
    flags = binding.SPEC_FLAG_VISITED_ONLY if args.visited_only else 0
    per_request = None
    if args.per_request:
        mix = [(0.0, 0, 1.0), (w.temperature, w.top_k, w.top_p), (1.0, 50, 1.0), (0.5, 0, 0.8)]
        per_request = (
            torch.tensor([mix[b % 4][0] for b in range(w.B)], dtype=torch.float32, device=dev),
            torch.tensor([mix[b % 4][1] for b in range(w.B)], dtype=torch.int32, device=dev),
            torch.tensor([mix[b % 4][2] for b in range(w.B)], dtype=torch.float32, device=dev))
    call = binding.PreparedVerify(inp["p"], inp["q"], tok, par, inp["max_depth"], w.temperature,
                                  w.top_k, w.top_p, seed=seed, offset=0, flags=flags,
                                  per_request=per_request)
    stream = torch.cuda.current_stream()
    clocks = clock_sampler(local)
    clocks.wait_first()
    t_warm0 = time.time()
    for _ in range(args.warmup):
        call()
    counters = call.read_counters()
    acc = call.out["accept_len"].cpu().numpy()
    tokens_per_step = int((acc + 1).sum())
    torch.cuda.synchronize()

    K = args.steps
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(K):
        call()  # one whole verify call: prepare, dense pass, walk
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    clocks.stop()
    elapsed_ms = ev0.elapsed_time(ev1)
    # the dense pass alone, each launch between two events (a separate loop: events
    # between the phases of the timed calls would keep the walk from starting while
    # the dense pass finishes)
    KR = min(K, 200)
    row_start = [torch.cuda.Event(enable_timing=True) for _ in range(KR)]
    row_end = [torch.cuda.Event(enable_timing=True) for _ in range(KR)]
    for k in range(KR):
        row_start[k].record(stream)
        call(binding.SPEC_PHASE_ROWS)
        row_end[k].record(stream)
    torch.cuda.synchronize()
    row_ms = [row_start[k].elapsed_time(row_end[k]) for k in range(KR)]
    row_avg_ms = sum(row_ms) / KR
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    rows_per_step = w.B * w.N
    value = whole_job_rate(world, rows_per_step, K, elapsed_ms)
    ms_per_step = elapsed_ms / K

    peaks, peak_kind = load_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    step_bytes = counters["dense_bytes"] + counters["walk_bytes"]
    # no dense pass ran: the visited-rows-only schedule, or a small vocabulary without a
    # cut (one warp per tree reads the rows it visits)
    no_dense = args.visited_only or counters["dense_rows"] == 0
    if no_dense:
        # the walk is the only kernel; its rows read over its time
        walk_ms = ms_per_step - row_avg_ms
        achieved = counters["walk_bytes"] / (walk_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak, "traffic": None,
                    "kernel": ("cluster_walk_kernel (visited rows only; latency-bound)"
                               if args.visited_only else
                               "small_walk_kernel (one warp per tree; latency-bound)"),
                    "peak_source": f"{peak_kind} hbm_gbs",
                    "algorithmic_bytes_per_launch": counters["walk_bytes"],
                    "avg_launch_ms": walk_ms}
    else:
        # The graded figure is the whole step's: the dense pass's bytes plus the walk's
        # (its visited rows' re-reads), over the step's time.  The row pass alone is
        # reported beside it.
        achieved = step_bytes / (ms_per_step / 1e3) / 1e9
        row_achieved = counters["dense_bytes"] / (row_avg_ms / 1e3) / 1e9
        # the committed captures are of the one-setting workload
        traffic, traffic_state = (None, None) if args.per_request else profiled_traffic(w.name)
        walk_traffic, walk_state = ((None, None) if args.per_request else
                                    profiled_traffic(w.name, "cluster_walk", WALK_SOURCES))
        row_pass = {"kernel": "row_pass_kernel (dense row pass)", "achieved": row_achieved,
                    "frac": row_achieved / hbm_peak, "avg_launch_ms": row_avg_ms,
                    "algorithmic_bytes_per_launch": counters["dense_bytes"], "traffic": traffic}
        if traffic_state == "stale":
            row_pass["traffic_note"] = "ncu capture predates the current row-pass sources"
        roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                    "frac": achieved / hbm_peak,
                    "traffic": (traffic + walk_traffic
                                if traffic is not None and walk_traffic is not None else None),
                    "kernel": "verify step: row_pass_kernel + cluster_walk_kernel",
                    "peak_source": f"{peak_kind} hbm_gbs",
                    "algorithmic_bytes_per_step": step_bytes,
                    "avg_step_ms": ms_per_step, "row_pass": row_pass}
        if walk_state != "current":
            roofline["traffic_note"] = ("no ncu capture of the walk on the current sources"
                                        if walk_state is None else
                                        "walk capture predates the current walk sources")

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "V": w.V, "logits": w.dtype,
                   "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p,
                   "tree": f"{w.tree}, depth {inp['max_depth']}, branching <= {w.max_branch}",
                   "rng_offset": "fixed per step",
                   "schedule": ("visited rows only (no dense pass)" if args.visited_only
                                else "one warp per tree, no dense pass (small vocabulary)"
                                if no_dense else "dense pass over every row"),
                   "sampling": ("per request: trees cycle through greedy, the workload's "
                                "setting, top-k 50 at T=1, top-p 0.8 at T=0.5"
                                if args.per_request else "one setting for every tree"),
                   "l2": f"inputs {2 * w.B * w.N * w.V * (2 if w.dtype == 'bf16' else 4) / 1e9:.2f}"
                         " GB per step, larger than L2; no flush",
                   "parallelism": f"weak: {world} rank(s) x {w.B} trees"},
        "tokens_per_s": whole_job_rate(world, tokens_per_step, K, elapsed_ms),
        "step_hbm_gbs": step_bytes / (ms_per_step / 1e3) / 1e9,
        "work_per_step": counters,
        "roofline": roofline,
        "gpu_launches": (1 if no_dense else 2) * K,  # [dense pass +] walk per call
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    result["clocks"]["warmup_and_timed"] = clocks.summary(t_warm0, t_wall1)

    if not args.no_e2e and not args.per_request:
        result["e2e"] = run_e2e(args, w, inp, dev, stream)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = run_cpu_baseline(args, w, inp)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_ours_lmhead(args, w, world, rank, local, dev):
    """The fused LM-head workload: every step computes the target logits of all B*N
    nodes from their features on the tensor cores (with the row statistics), the draft
    rows' statistics, and the walk.  The roofline is the LM-head GEMM's FLOP rate."""
    from speculative_decoding_tree_spec_gb300 import binding

    seed = shard_seed(args.seed, rank)
    inp = wl.build_lmhead_inputs(w, seed, device=dev)
    tok = torch.as_tensor(inp["tokens"], device=dev)
    par = torch.as_tensor(inp["parents"], device=dev)
    args_ = (inp["features"], inp["weight"], inp["q"], tok, par, inp["max_depth"], w.temperature,
             w.top_k, w.top_p)
    first = binding.verify_tree_fused_lmhead(*args_, seed=seed, want_counters=True)
    out = {k: v for k, v in first.items() if torch.is_tensor(v)}
    ws = torch.empty(max(256, int(binding.lib().spec_fused_lmhead_workspace_size(w.B, w.N, w.V))),
                     dtype=torch.uint8, device=dev)
    counters = first["counters"]

    def call(phases):
        binding.verify_tree_fused_lmhead(*args_, seed=seed, out=out, workspace=ws, phases=phases)

    stream = torch.cuda.current_stream()
    clocks = clock_sampler(local)
    clocks.wait_first()
    t_warm0 = time.time()
    for _ in range(args.warmup):
        call(binding.SPEC_PHASE_ALL_FUSED)
    acc = out["accept_len"].cpu().numpy()
    tokens_per_step = int((acc + 1).sum())
    torch.cuda.synchronize()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gs = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ge = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ev0.record(stream)
    for k in range(K):
        call(binding.SPEC_PHASE_PREPARE)
        gs[k].record(stream)
        call(binding.SPEC_PHASE_LMHEAD)
        ge[k].record(stream)
        call(binding.SPEC_PHASE_ROWS | binding.SPEC_PHASE_WALK)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    clocks.stop()
    elapsed_ms = max_over_ranks(ev0.elapsed_time(ev1), world, dev)
    gemm_ms = sum(gs[k].elapsed_time(ge[k]) for k in range(K)) / K
    d = inp["features"].shape[1]
    flops = 2.0 * w.B * w.N * w.V * d
    peaks, peak_kind = load_peaks()
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    achieved = flops / (gemm_ms / 1e3) / 1e12
    result = {
        "metric": METRIC, "value": whole_job_rate(world, w.B * w.N, K, elapsed_ms), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": elapsed_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "N": w.N, "V": w.V, "d": d, "logits": "bf16",
                   "temperature": w.temperature, "top_k": w.top_k, "top_p": w.top_p,
                   "tree": f"{w.tree}, depth {inp['max_depth']}, branching <= {w.max_branch}",
                   "l2": f"weight {w.V * d * 2 / 1e9:.2f} GB + logits written "
                         f"{w.B * w.N * w.V * 2 / 1e9:.2f} GB per step, larger than L2; no flush",
                   "parallelism": f"weak: {world} rank(s) x {w.B} trees"},
        "tokens_per_s": whole_job_rate(world, tokens_per_step, K, elapsed_ms),
        "work_per_step": counters,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "lmhead_kernel (tcgen05 GEMM + row statistics) + combine",
                     "peak_source": f"{peak_kind} bf16_tflops_sustained",
                     "algorithmic_flops_per_launch": flops, "avg_launch_ms": gemm_ms},
        "gpu_launches": 4 * K if w.temperature > 0 else 3 * K,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    result["clocks"]["warmup_and_timed"] = clocks.summary(t_warm0, t_wall1)
    if not args.no_e2e:
        host = {"features": inp["features"].cpu().pin_memory(),
                "q": inp["q"].cpu().pin_memory(),
                "tokens": torch.as_tensor(inp["tokens"]).pin_memory(),
                "parents": torch.as_tensor(inp["parents"]).pin_memory()}
        dbuf = {"features": torch.empty_like(inp["features"]), "q": torch.empty_like(inp["q"]),
                "tokens": torch.empty_like(tok), "parents": torch.empty_like(par)}
        outs = {k: torch.empty(out[k].shape, dtype=out[k].dtype).pin_memory()
                for k in ("accept_len", "tokens", "path")}

        def step():
            for k, v in host.items():
                dbuf[k].copy_(v, non_blocking=True)
            binding.verify_tree_fused_lmhead(dbuf["features"], inp["weight"], dbuf["q"],
                                             dbuf["tokens"], dbuf["parents"], inp["max_depth"],
                                             w.temperature, w.top_k, w.top_p, seed=seed, out=out,
                                             workspace=ws)
            for k, v in outs.items():
                v.copy_(out[k], non_blocking=True)

        for _ in range(2):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1) / args.e2e_steps, world, dev)
        result["e2e"] = {"value": world * w.B * w.N / (ms / 1e3), "unit": UNIT,
                         "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host.values()),
                         "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in outs.values()),
                         "ms_per_step": ms, "steps": args.e2e_steps}
    if rank == 0:
        print(json.dumps(result), flush=True)
    return result


def run_commit(args):
    """The accepted-path commit on a KV cache shaped like an 8B model's (32 layers x K/V
    = 64 planes, 8 heads x 128 x bf16 = 2 KB per position), after verifying the
    workload's trees: the bytes it moves (read + write) per second."""
    from speculative_decoding_tree_spec_gb300 import binding

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    seed = shard_seed(args.seed, rank)
    inp = wl.build_inputs(w, seed=seed, device=dev)
    out = binding.verify_tree(inp["p"], inp["q"], torch.as_tensor(inp["tokens"], device=dev),
                              torch.as_tensor(inp["parents"], device=dev), inp["max_depth"],
                              w.temperature, w.top_k, w.top_p, seed=seed)
    planes, row_elems, n_pos = 64, 1024, 1024 + w.N
    cache = torch.zeros((planes, w.B, n_pos, row_elems), dtype=torch.bfloat16, device=dev)
    prefix = torch.full((w.B,), 1024, dtype=torch.int32, device=dev)
    acc = out["accept_len"]
    moved = int(acc.clamp(min=0).sum().item()) * planes * row_elems * 2 * 2
    # one launch per step, replayed from a CUDA graph (a plain Python call per launch
    # would time the host, not the kernel)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            binding.commit_accepted_path(cache, prefix, out["path"], acc)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        binding.commit_accepted_path(cache, prefix, out["path"], acc)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    peaks, peak_kind = load_peaks()
    gbs = moved / (ms / 1e3) / 1e9
    line = {"metric": "accepted-path commit: cache bytes moved (read + write) per second",
            "value": world * moved / (ms / 1e3), "unit": "B/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": w.name, "cache": f"{planes} planes x {w.B} sequences x {n_pos} "
                       f"positions x {row_elems * 2} B", "accepted_nodes": int(acc.clamp(min=0).sum())},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                         "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                         "kernel": "commit_kernel", "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": moved, "avg_launch_ms": ms},
            "timing": "CUDA graph replay of the launch; the cache lives on the device",
            "gpu_launches": args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_tree(args):
    """The EAGLE-2 dynamic draft tree for the workload's batch: the draft model's
    candidates in the method's usual setting (10 children per expanded node, 10 nodes
    expanded per layer, 6 layers: 510 candidates), one expansion top-k per layer that
    feeds the next, then the rerank to the workload's N nodes, flattening and the
    ancestor mask.  Drafts built per second."""
    from speculative_decoding_tree_spec_gb300 import binding

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    layers, ek, ch = 6, 10, 10
    d = wl.make_draft_candidates(w.B, layers=layers, expand_k=ek, children=ch,
                                 seed=shard_seed(args.seed, rank))
    par, tok, prob, root = (torch.from_numpy(x).to(dev) for x in (d.parent, d.token, d.prob, d.root))
    n, m = d.parent.shape[1], w.N - 1
    bounds = [(0, ch)] + [(ch + i * ek * ch, ch + (i + 1) * ek * ch) for i in range(layers - 2)]

    def step():
        for lo, hi in bounds:
            binding.tree_expand_topk(par, prob, lo, hi, ek)
        return binding.tree_build(par, tok, prob, root, m)

    # the step's launches go through a CUDA graph (six tiny launches: host-bound
    # otherwise); the e2e figure below is the plain call path with host buffers
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(args.warmup):
            step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps

    # end to end: candidates from pinned host memory in, the draft back out, every step
    host = [torch.from_numpy(x).pin_memory() for x in (d.parent, d.token, d.prob, d.root)]
    dbuf = [h.to(dev) for h in host]

    def e2e_step():
        for h, x in zip(host, dbuf):
            x.copy_(h, non_blocking=True)
        for lo, hi in bounds:
            binding.tree_expand_topk(dbuf[0], dbuf[2], lo, hi, ek)
        out = binding.tree_build(*dbuf, m)
        return {k: v.to("cpu", non_blocking=True) for k, v in out.items()}

    for _ in range(3):
        res = e2e_step()
    torch.cuda.synchronize()
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = sum(v.numel() * v.element_size() for v in res.values())
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.e2e_steps
    peaks, peak_kind = load_peaks()
    M = m + 1
    # per tree: the candidate list read by each expansion (parents + confidences of the
    # chains it walks, counted once) and by the build (parents, tokens, confidences),
    # plus the draft written (4 int32 arrays + the mask)
    bytes_step = w.B * (len(bounds) * n * 8 + n * 12 + M * 16 + M * M)
    gbs = bytes_step / (ms / 1e3) / 1e9
    line = {"metric": "EAGLE-2 draft trees built (expand + rerank + flatten + mask) per second",
            "value": world * w.B / (ms / 1e3), "unit": "trees/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"eagle2_tree_b{w.B}_n{n}_m{m}", "candidates": n,
                       "draft_nodes": M, "expansions_per_step": len(bounds)},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                         "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "traffic": None,
                         "kernel": "tree_expand_kernel + tree_build_kernel (whole step)",
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": bytes_step, "avg_launch_ms": ms,
                         "note": "latency-bound: a few KB per tree, one CTA per tree"},
            "e2e": {"value": world * w.B / (e2e_ms / 1e3), "unit": "trees/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "timing": "CUDA graph replay of the step; inputs resident, outputs left in HBM",
            "gpu_launches": args.steps * (len(bounds) + 1)}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_draft(args):
    """Draft-side top-k drafting: the rows of the nodes one EAGLE-2 layer expands (the
    workload's batch x 10 expanded nodes) of draft logits over the workload's vocabulary
    (bf16, N(0, 3^2)), the 10 children and confidences of each at T = 1.  Rows per second
    and the HBM roofline of the one kernel."""
    from speculative_decoding_tree_spec_gb300 import binding

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    R, V, k = w.B * 10, w.V, 10
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(args.seed, rank))
    logits = wl.empty_rows((R, V), torch.bfloat16, dev)
    logits.copy_(torch.randn((R, V), generator=g, device=dev) * 3)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        binding.draft_topk(logits, k, 1.0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        binding.draft_topk(logits, k, 1.0)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps

    # end to end: the rows from pinned host memory in, children and confidences back
    host = logits.cpu().pin_memory()
    dbuf = torch.empty_like(logits)

    def e2e_step():
        dbuf.copy_(host, non_blocking=True)
        out = binding.draft_topk(dbuf, k, 1.0)
        return {a: v.to("cpu", non_blocking=True) for a, v in out.items()}

    for _ in range(2):
        res = e2e_step()
    torch.cuda.synchronize()
    h2d = host.numel() * host.element_size()
    d2h = sum(v.numel() * v.element_size() for v in res.values())
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.e2e_steps
    peaks, peak_kind = load_peaks()
    bytes_launch = R * V * 2
    gbs = bytes_launch / (ms / 1e3) / 1e9
    traffic, _ = profiled_traffic(f"r{R}_v{V}_k{k}", "draft_topk", DRAFT_SOURCES)
    line = {"metric": "draft-side top-k drafting: expanded-node rows per second",
            "value": world * R / (ms / 1e3), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"draft_topk_r{R}_v{V}_k{k}", "rows": R, "V": V, "k": k,
                       "temperature": 1.0, "l2": f"rows {bytes_launch / 1e6:.0f} MB, larger than L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": float(peaks["hbm_gbs"]),
                         "unit": "GB/s", "frac": gbs / float(peaks["hbm_gbs"]), "traffic": traffic,
                         "kernel": "draft_topk_kernel", "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": bytes_launch, "avg_launch_ms": ms},
            "e2e": {"value": world * R / (e2e_ms / 1e3), "unit": "rows/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_draft_fused(args):
    """Draft LM head + top-k in one call: the features of the nodes one EAGLE-2 layer
    expands (the workload's batch x 10, d = 4096, N(0, 1)) times a draft LM-head weight
    (V x 4096, N(0, 0.02^2)) on the tensor cores, the bf16 logits ranked by the top-k
    kernel (k = 10, T = 1).  Rows per second and the tensor roofline of the call."""
    from speculative_decoding_tree_spec_gb300 import binding

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    w = wl.WORKLOADS[args.workload]
    if args.batch:
        w = w.with_(B=args.batch)
    R, V, d, k = w.B * 10, w.V, 4096, 10
    g = torch.Generator(device=dev)
    g.manual_seed(shard_seed(args.seed, rank))
    feats = torch.randn((R, d), generator=g, device=dev).to(torch.bfloat16)
    weight = (torch.randn((V, d), generator=g, device=dev) * 0.02).to(torch.bfloat16)
    ws = torch.empty(int(binding.lib().spec_draft_fused_workspace_size(R, V, k)), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        binding.draft_topk_fused_lmhead(feats, weight, k, 1.0, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    e0.record(stream)
    for _ in range(args.steps):
        binding.draft_topk_fused_lmhead(feats, weight, k, 1.0, workspace=ws)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps

    # end to end: the features from pinned host memory in, children and confidences back
    # (the weight stays resident, as a model's weights do)
    host = feats.cpu().pin_memory()
    dbuf = torch.empty_like(feats)

    def e2e_step():
        dbuf.copy_(host, non_blocking=True)
        out = binding.draft_topk_fused_lmhead(dbuf, weight, k, 1.0, workspace=ws)
        return {a: v.to("cpu", non_blocking=True) for a, v in out.items()}

    for _ in range(2):
        res = e2e_step()
    torch.cuda.synchronize()
    h2d = host.numel() * host.element_size()
    d2h = sum(v.numel() * v.element_size() for v in res.values())
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), world, dev) / args.e2e_steps
    peaks, peak_kind = load_peaks()
    flops = 2.0 * R * V * d
    tf = flops / (ms / 1e3) / 1e12
    peak = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    line = {"metric": "draft LM head + top-k drafting in one call: expanded-node rows per second",
            "value": world * R / (ms / 1e3), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"draft_lmhead_topk_r{R}_v{V}_d{d}_k{k}", "rows": R, "V": V,
                       "d": d, "k": k, "temperature": 1.0,
                       "logits": "bf16 rows in the workspace, read back by the ranking kernel"},
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s",
                         "frac": tf / peak, "traffic": None,
                         "kernel": "lmhead_kernel + draft_topk_kernel (whole call)",
                         "peak_source": f"{peak_kind} bf16_tflops_sustained",
                         "algorithmic_flops_per_launch": flops, "avg_launch_ms": ms},
            "e2e": {"value": world * R / (e2e_ms / 1e3), "unit": "rows/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps * 2}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, w, inp, dev, stream):
    """The same metric through the public C-ABI call with host buffers: every step
    copies the inputs host->device from pinned memory, verifies, and copies the
    accepted lengths, tokens and paths back."""
    from speculative_decoding_tree_spec_gb300 import binding

    host = {k: inp[k].cpu().pin_memory() for k in ("p", "q")}
    host["tokens"] = torch.as_tensor(inp["tokens"]).pin_memory()
    host["parents"] = torch.as_tensor(inp["parents"]).pin_memory()
    dbuf = {k: torch.empty_like(v, device=dev) for k, v in host.items()}
    flags = binding.SPEC_FLAG_VISITED_ONLY if args.visited_only else 0
    call = binding.PreparedVerify(dbuf["p"], dbuf["q"], dbuf["tokens"], dbuf["parents"],
                                  inp["max_depth"], w.temperature, w.top_k, w.top_p, seed=1, offset=0,
                                  flags=flags)
    outs = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
            for k, v in call.out.items() if k in ("accept_len", "tokens", "path")}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())

    def step():
        for k, v in host.items():
            dbuf[k].copy_(v, non_blocking=True)
        call()
        for k, v in outs.items():
            v.copy_(call.out[k], non_blocking=True)

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.e2e_steps
    world = dist_env()[0]
    ms = max_over_ranks(ms, world, dev)
    return {"value": world * w.B * w.N / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": args.e2e_steps}


def run_cpu_baseline(args, w, inp):
    import oracle

    oracle.build()
    n_pool = min(16, w.B)
    idx = torch.arange(n_pool, device=inp["p"].device)
    pool = {"p": wl.host_logits(inp["p"].index_select(0, idx)),
            "q": wl.host_logits(inp["q"].index_select(0, idx)),
            "tokens": inp["tokens"][:n_pool], "parents": inp["parents"][:n_pool],
            "max_depth": inp["max_depth"]}
    threads = args.host_threads or os.cpu_count() or 1
    wall, rows = time_oracle(w, pool, args.cpu_trees, threads, args.seed)
    return {"value": rows / wall, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{args.cpu_trees} tree-steps cycling over the first {n_pool} trees of "
                      f"the timed batch ({w.name}), one tree per host thread task"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.op == "commit":
        run_commit(args)
    elif args.op == "tree":
        run_tree(args)
    elif args.op == "draft" and args.fused:
        run_draft_fused(args)
    elif args.op == "draft":
        run_draft(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
