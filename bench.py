#!/usr/bin/env python
"""Throughput of one DSpark draft-verify cycle (propose -> schedule -> verify)
for a whole serving batch on one GB300, through the C ABI.

Default workload: R = 256 requests, gamma = 7, V = 151936, Markov rank 256,
bf16 tables, greedy, SPS(B) flat at 1e3 steps/s up to B = 256 then ~1/B
(1024 entries).  Inputs are seeded synthetic tensors resident in HBM; each
timed step is one cycle, captured as a single CUDA graph and bracketed by
CUDA events on the launching stream; L2 is flushed (a 512 MB write) between
steps, outside the events.  The cycle is the library's one-call dsd_cycle,
which runs the schedule inside the proposal's last launch.  A second pass
replays dsd_propose, dsd_schedule and dsd_verify as one graph each, with an
event between them, for the phase breakdown and the propose roofline.

Prints ONE JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
the host cores on bounded samples of the same workload instead.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "draft-verify cycles/sec and tokens/sec at V=151936,γ=7,R=256; % of HBM roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "simt_bias_kernel": ["propose_simt.cu", "dsd_common.cuh"],
    "propose_tc_kernel": ["propose_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "dsd_common.cuh"],
    "propose_tc_pair_kernel": ["propose_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "dsd_common.cuh"],
    "residual_tc_kernel": ["propose_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "dsd_common.cuh"],
    "propose_mma_kernel": ["propose_mma.cu", "dsd_common.cuh"],
    "verify_rows": ["verify.cu", "dsd_common.cuh"],
    "overlap_split": ["overlap.cu", "tc_common.cuh", "tc_ptx.cuh", "dsd_common.cuh"],
    "confidence_head_kernel": ["confidence.cu", "dsd_common.cuh"],
    "loss_tc_kernel": ["loss_tc.cu", "tc_common.cuh", "tc_ptx.cuh", "dsd_common.cuh"],
}
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def dist_info():
    return env_int("RANK", 0), env_int("LOCAL_RANK", 0), env_int("WORLD_SIZE", 1)


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def source_hash(kernel: str) -> str:
    """Hash of a kernel's source files with comments and blank space removed,
    so that only a change of the code voids the stored counters."""
    import re

    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, []):
        with open(os.path.join(ROOT, "semi_autoregressive_draft_gb300", "csrc", f),
                  encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode("utf-8"))
    return h.hexdigest()[:16]


def traffic_for(kernel: str, workload: str):
    """DRAM bytes (read + write) per roofline unit from the committed ncu
    summary, or None when the kernel source changed since the counters were
    taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            table = json.load(f)
    except (OSError, ValueError):
        return None
    ent = table.get(kernel, {}).get(workload)
    if not ent or ent.get("source_hash") != source_hash(kernel):
        return None
    return ent.get("dram_bytes")


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["--id=" + self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summary()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_uuid(device_index: int):
    import torch

    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# --------------------------------------------------------------- workloads

def cycle_spec(name):
    from semi_autoregressive_draft_gb300 import synth

    return synth.CYCLE_SPECS[name]


def workload_label(spec):
    mode = "greedy" if spec.temperature == 0 else f"sampled T={spec.temperature:g}"
    return (f"{spec.name}: R={spec.R} gamma={spec.G} V={spec.V} r={spec.r} {spec.dtype} "
            f"{mode}, SPS {spec.sps_kind}")


def propose_step_bytes(spec):
    """Bytes one draft-step launch must move: the U rows of its position, all
    of the projection W (every step projects onto the whole vocabulary, and
    the step before evicts most of it from L2 while streaming its own U
    rows), the gathered E rows and the argmax keys."""
    esz = 2 if spec.dtype == "bf16" else 4
    R, V, r = spec.R, spec.V, spec.r
    return R * V * esz + V * r * esz + R * r * esz + R * 8


def propose_alg_bytes(spec):
    """Bytes of the propose phase with W counted once per draft step: gamma
    step launches plus the confidences, previous tokens and the four
    [R, gamma] outputs."""
    R, G = spec.R, spec.G
    return G * propose_step_bytes(spec) + R * G * 4 + R * 4 + 4 * R * G * 4


def tensor_report(spec, phase_s, engine):
    """The bias GEMM's throughput over the propose phase: 2 R r V flops per
    draft step, gamma steps, against the measured bf16 peak (sustained: the
    phase runs inside a long timed loop).  Only the tensor-core engines run
    it on tensor cores."""
    flops = 2.0 * spec.R * spec.r * spec.V * spec.G
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        peak, kind = float(pk["bf16_tflops_sustained"]), "measured sustained"
    except (OSError, ValueError, KeyError):
        peak, kind = 1700.0, "fallback sustained"
    achieved = flops / phase_s / 1e12
    return {"engine": engine, "flops_per_phase": flops, "achieved_tflops": achieved,
            "peak_tflops": peak, "peak_kind": f"{kind} (MEASURED_PEAKS.json bf16)",
            "frac": achieved / peak}


def fma_report(flops, phase_s, engine):
    """The CUDA-core engine's inner products (2 R r V flops per draft step) on
    the fp32 FMA pipes, against their peak derived from unit counts and the
    clock: SMs x 128 fp32 lanes x 2 flops x the maximum SM clock
    (MEASURED_PEAKS.json sm_max_mhz, else 2070 MHz).  At R = 16 this work,
    not the table bytes, bounds the engine: 1.24 GFLOP per step is 15 us at
    the peak against 12 us for its 82.7 MB at the measured copy rate."""
    import torch

    try:
        with open(PEAKS_FILE) as f:
            mhz, kind = float(json.load(f)["sm_max_mhz"]), "MEASURED_PEAKS.json sm_max_mhz"
    except (OSError, ValueError, KeyError):
        mhz, kind = 2070.0, "nominal maximum SM clock"
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    peak = sms * 128 * 2 * mhz * 1e6 / 1e12
    achieved = flops / phase_s / 1e12
    return {"engine": engine, "bound": "alu", "flops": flops, "achieved_tflops": achieved,
            "peak_tflops": peak, "frac": achieved / peak,
            "peak_kind": f"derived: {sms} SMs x 128 fp32 lanes x 2 x {mhz:.0f} MHz ({kind})"}


def propose_w_once_bytes(spec):
    """The phase's compulsory bytes: every U row once and W once for the
    whole phase (the lower bound if W stayed in L2 across the steps)."""
    esz = 2 if spec.dtype == "bf16" else 4
    R, G, V, r = spec.R, spec.G, spec.V, spec.r
    return (R * G * V * esz + V * r * esz + R * G * r * esz + R * G * 4 + R * 4
            + 4 * R * G * 4)


def verify_alg_bytes(spec, B):
    esz = 2 if spec.dtype == "bf16" else 4
    return B * spec.V * esz


# --------------------------------------------------------------- CPU oracle
# The fp64 oracle is timed in worker processes started with "spawn" (never
# forked: the parent may already hold a CUDA context), each with
# single-threaded BLAS, so that "cores" is the number of workers that really
# ran.  The inputs reach the workers as memory-mapped .npy files in a
# temporary directory (shared page cache, no per-worker copy): the bf16 logit
# rows as their raw 16-bit patterns, widened exactly to fp32 in the worker,
# and E, W widened once to fp64 (the oracle's precision).

_POOL_ARRAYS = {}
_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _pool_init(dirpath):
    import numpy as np

    for k in ("U", "P", "E", "W", "conf", "prev_tok", "req_id"):
        _POOL_ARRAYS[k] = np.load(os.path.join(dirpath, k + ".npy"), mmap_mode="r")


def _pool_rows(a, idx):
    import numpy as np

    rows = np.asarray(a[idx])
    if rows.dtype == np.uint16:          # bf16 bit patterns -> fp32, exactly
        rows = (rows.astype(np.uint32) << 16).view(np.float32)
    return rows


def _pool_requests(job):
    """Propose + verify of some requests of the batch (one worker)."""
    import numpy as np

    from oracle import dsd_oracle as O

    idx, keep, temperature, seed = job
    h = _POOL_ARRAYS
    idx = np.asarray(idx)
    t0 = time.perf_counter()
    rid = np.asarray(h["req_id"][idx]).astype(np.int64)
    U = _pool_rows(h["U"], idx)
    P = _pool_rows(h["P"], idx)
    prev = np.asarray(h["prev_tok"][idx])
    prop = O.propose(U, h["E"], h["W"], np.asarray(h["conf"][idx]), prev, rid, temperature, seed)
    ver = O.verify(P, U, h["E"], h["W"], prev, prop["tokens"], np.asarray(keep), rid,
                   temperature, seed)
    return time.perf_counter() - t0, ver["accept_len"].tolist()


class OraclePool:
    """Times full draft-verify cycles of the fp64 oracle on the host cores."""

    def __init__(self, spec, x, workers=None):
        import tempfile

        import numpy as np

        from oracle import dsd_oracle as O
        from semi_autoregressive_draft_gb300 import synth

        self.spec = spec
        self.workers = max(1, workers or os.cpu_count() or 1)
        self.seed = x["seed"]
        self.dir = tempfile.mkdtemp(prefix="dsd_oracle_")
        for k in ("U", "P"):
            t = x[k].detach()
            a = (t.view(dtype=__import__("torch").int16).cpu().numpy().view(np.uint16)
                 if spec.dtype == "bf16" else t.float().cpu().numpy())
            np.save(os.path.join(self.dir, k + ".npy"), a)
        for k in ("E", "W"):
            np.save(os.path.join(self.dir, k + ".npy"), synth.to_numpy(x[k]).astype(np.float64))
        for k in ("conf", "prev_tok", "req_id"):
            np.save(os.path.join(self.dir, k + ".npy"), synth.to_numpy(x[k]))
        self.conf = synth.to_numpy(x["conf"])
        self.sps = synth.to_numpy(x["sps"])
        self._O = O
        self._pools = {}

    def _pool(self, n):
        import multiprocessing as mp

        if n not in self._pools:
            saved = {k: os.environ.get(k) for k in _BLAS_ENV}
            for k in _BLAS_ENV:
                os.environ[k] = "1"
            try:
                pool = mp.get_context("spawn").Pool(n, initializer=_pool_init,
                                                    initargs=(self.dir,))
                pool.map(abs, range(n))           # every worker has started
            finally:
                for k, v in saved.items():
                    if v is None:
                        os.environ.pop(k, None)
                    else:
                        os.environ[k] = v
            self._pools[n] = pool
        return self._pools[n]

    def schedule(self):
        O = self._O
        surv = O.survival(self.conf).astype("float32")
        return O.schedule(surv, self.sps)["keep_len"]

    def cycle(self, reqs=None, workers=None):
        """One cycle (schedule of the whole batch, then propose + verify of
        `reqs`, default all requests) on `workers` processes; returns (wall
        seconds, committed tokens of those requests, CPU seconds in workers)."""
        R = self.spec.R
        reqs = list(range(R)) if reqs is None else list(reqs)
        n = workers or self.workers
        pool = self._pool(n)
        chunk = max(1, len(reqs) // (4 * n))
        t0 = time.perf_counter()
        keep = self.schedule()
        jobs = [(reqs[i:i + chunk], keep[reqs[i:i + chunk]], self.spec.temperature, self.seed)
                for i in range(0, len(reqs), chunk)]
        res = pool.map(_pool_requests, jobs, chunksize=1)
        wall = time.perf_counter() - t0
        tokens = sum(a + 1 for _, acc in res for a in acc)
        return wall, tokens, sum(t for t, _ in res)

    def single_thread(self, n_req):
        """Per-request time of one single-threaded worker over n_req requests,
        extrapolated to the whole batch (plus the measured schedule)."""
        self.cycle(reqs=[0], workers=1)            # warm the worker
        t0 = time.perf_counter()
        self.schedule()
        t_sched = time.perf_counter() - t0
        wall, _, _ = self.cycle(reqs=range(n_req), workers=1)
        per_req = (wall - t_sched) / n_req
        return t_sched + per_req * self.spec.R, wall

    def close(self):
        import shutil

        for pool in self._pools.values():
            pool.close()
            pool.join()
        self._pools = {}
        shutil.rmtree(self.dir, ignore_errors=True)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def oracle_baseline(spec, x, n_cycles=2, n_single=8):
    """The in-run CPU baseline: n_cycles full-batch cycles on every host core
    (after one untimed cycle), measured, plus a single-thread figure."""
    with OraclePool(spec, x) as pool:
        pool.cycle()
        runs = [pool.cycle() for _ in range(n_cycles)]
        st_est, st_wall = pool.single_thread(min(n_single, spec.R))
        wall = statistics.mean(w for w, _, _ in runs)
        busy = sum(c for _, _, c in runs)
        return {
            "value": 1.0 / wall, "unit": "cycles/s", "cores": pool.workers, "kind": "oracle",
            "sample": (f"{n_cycles} full cycles of the whole batch (schedule of all {spec.R} "
                       f"requests, then propose + verify of every request, all {spec.G} "
                       f"positions, full V={spec.V}) on {pool.workers} single-threaded worker "
                       f"processes, after one untimed cycle; measured, not extrapolated"),
            "ms_per_cycle": wall * 1e3,
            "cpu_seconds": busy,
            "single_thread": {
                "value": 1.0 / st_est, "unit": "cycles/s", "cores": 1,
                "sample": (f"propose + verify of {min(n_single, spec.R)} requests on one "
                           f"single-threaded process ({st_wall:.1f} s measured) plus the "
                           f"measured schedule, extrapolated linearly to {spec.R} requests"),
            },
        }


def cycle_config(spec, world):
    """The config dict both arms print for a draft-verify workload."""
    return {"workload": workload_label(spec), "R": spec.R, "gamma": spec.G, "V": spec.V,
            "rank": spec.r, "temperature": spec.temperature, "parallelism": f"replicas x{world}",
            "l2": f"inputs {cycle_input_bytes(spec) / 1e9:.2f} GB; the GPU arm flushes L2 "
                  f"(512 MB write outside the events) between steps"}


def cycle_input_bytes(spec):
    esz = 2 if spec.dtype == "bf16" else 4
    return (spec.R * spec.G + spec.R * (spec.G + 1)) * spec.V * esz + 2 * spec.V * spec.r * esz


# --------------------------------------------------------------------- arms

def run_reference(args):
    """The oracle arm: each step is one full draft-verify cycle of the whole
    batch (schedule, then propose + verify of every request) on the host
    cores, timed on the wall clock; nothing is extrapolated."""
    rank, local_rank, world = dist_info()
    if rank != 0:
        return 0
    from semi_autoregressive_draft_gb300 import synth

    spec = cycle_spec(args.workload)
    x = synth.cycle_inputs(spec, device="cpu")
    n_req = spec.R if args.ref_requests <= 0 else min(args.ref_requests, spec.R)
    with OraclePool(spec, x) as pool:
        for s in range(args.warmup):
            pool.cycle(reqs=[(s * 37 + i) % spec.R for i in range(n_req)])
        times, toks = [], []
        for s in range(args.steps):
            wall, tok, _ = pool.cycle(reqs=[(s * 37 + i) % spec.R for i in range(n_req)])
            times.append(wall)
            toks.append(tok)
        st_est, st_wall = pool.single_thread(min(8, spec.R))
        workers = pool.workers
    sec = statistics.mean(times)
    frac = n_req / spec.R
    value = frac / sec                     # whole-batch cycles per second
    if n_req == spec.R:
        sample = (f"each step: one full cycle of the whole batch (schedule of all {spec.R} "
                  f"requests, then propose + verify of every request, all {spec.G} positions, "
                  f"full V={spec.V}) on {workers} single-threaded worker processes; measured")
    else:
        sample = (f"each step: schedule of all {spec.R} requests, then propose + verify of "
                  f"{n_req} of them on {workers} single-threaded worker processes; value = "
                  f"{n_req}/{spec.R} of a cycle per measured step time")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "cycles/s",
        "tokens_per_s": statistics.mean(toks) / frac * value if toks else None,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cycle_config(spec, world),
        "cpu_baseline": {"value": value, "unit": "cycles/s", "cores": workers, "kind": "oracle",
                         "sample": sample,
                         "single_thread": {"value": 1.0 / st_est, "unit": "cycles/s",
                                           "cores": 1,
                                           "sample": f"propose + verify of {min(8, spec.R)} "
                                                     f"requests on one process ({st_wall:.1f} s "
                                                     f"measured), extrapolated to {spec.R}"}},
        "e2e": {"value": value, "unit": "cycles/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "notes": "fp64 numpy oracle on the host cores; no GPU involved",
    }
    print(json.dumps(line), flush=True)
    return 0


def run_overlap(args, dsd, synth, dev, world):
    """The offline overlap call on the full teacher-forced workload (4096 blocks
    x gamma positions over the whole vocabulary); inputs (17 GB) exceed L2."""
    import numpy as np
    import torch

    spec = synth.OverlapSpec(N=args.blocks) if args.blocks else synth.OverlapSpec()
    ox = synth.overlap_inputs(spec, device=dev)
    ctx = dsd.Context(spec.V, 64, spec.G, 8, dtype="bf16", device=dev.index)
    stream = torch.cuda.Stream(device=dev)
    out = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            out = ctx.overlap(ox["P"], ox["Q"], ox["valid_len"], out=out)
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    c0 = ctx.launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(dev.index))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    with torch.cuda.stream(stream):
        for e in evs:
            e[0].record(stream)
            out = ctx.overlap(ox["P"], ox["Q"], ox["valid_len"], out=out)
            e[1].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    assert ctx.sync_status(stream) == 0
    launches = ctx.launch_count() - c0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    vl = ox["valid_len"].cpu().numpy()
    valid_rows = int(np.clip(vl, 0, spec.G).sum())
    alg = valid_rows * 2 * spec.V * 2 + spec.N * spec.G * 8 + spec.N * 4
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": f"overlap blocks/s (a = sum min(p, q), tau_prob) at N={spec.N}, gamma={spec.G}, "
                  f"V={spec.V}",
        "value": world * spec.N / (ms / 1e3), "unit": "blocks/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "fp32", "data": "synthetic",
        "config": {"workload": f"overlap: N={spec.N} gamma={spec.G} V={spec.V} bf16, "
                               f"{spec.ragged_frac:.0%} ragged blocks",
                   "valid_rows": valid_rows, "l2": f"inputs {2 * spec.N * spec.G * spec.V * 2 / 1e9:.1f} GB, larger than L2"},
        "roofline": {"bound": "hbm", "kernel": "overlap_split", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic_for("overlap_split", "overlap"),
                     "alg_bytes": alg, "per": "one overlap call",
                     "alg_bytes_note": "valid P and Q rows once + a, l1 [N, gamma] + valid_len"},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches, "clocks": clk,
    }
    ctx.close()
    return line


def run_loss(args, dsd, synth, dev, world):
    """The teacher-forced DSpark loss forward on one training sample's anchors
    (512 blocks x gamma positions, full vocabulary); inputs (2.2 GB) exceed L2.
    One call is two launches of loss_tc_kernel (normalisers, then L1) and a
    one-CTA fp64 finalize."""
    import torch

    spec = synth.LossSpec()
    x = synth.loss_inputs(spec, device=dev)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.B, dtype="bf16", device=dev.index)
    stream = torch.cuda.Stream(device=dev)
    args_ = (x["U"], x["E"], x["W"], x["prev_tok"], x["P"], x["target"], x["conf_logit"])
    out = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            out = ctx.loss_forward(*args_, out=out, stream=stream)
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    c0 = ctx.launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(dev.index))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    with torch.cuda.stream(stream):
        for e in evs:
            e[0].record(stream)
            out = ctx.loss_forward(*args_, out=out, stream=stream)
            e[1].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    assert ctx.sync_status(stream) == 0
    launches = ctx.launch_count() - c0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    rows = spec.B * spec.G
    # per launch of loss_tc_kernel: U and P rows once, W once, the E rows, the
    # per-row inputs and the partials it writes
    per_pass = (2 * rows * spec.V * 2 + spec.V * spec.r * 2 + rows * spec.r * 2
                + rows * 12 + rows * 16 * 5)
    peak, peak_kind = hbm_peak()
    # the two passes take all but the finalize's few microseconds of the call
    achieved = 2 * per_pass / (ms / 1e3) / 1e9
    line = {
        "metric": "teacher-forced DSpark loss rows/s (CE + L1 + confidence BCE, Markov bias "
                  "on tcgen05) at B=512 blocks, gamma=7, V=151936, rank 256",
        "value": world * rows / (ms / 1e3), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "fp32 (fp64 finalize)", "data": "synthetic",
        "config": {"workload": f"loss: B={spec.B} gamma={spec.G} V={spec.V} rank={spec.r} bf16",
                   "rows": rows, "l2": "inputs 2.2 GB, larger than L2"},
        "roofline": {"bound": "hbm", "kernel": "loss_tc_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": traffic_for("loss_tc_kernel", "loss"),
                     "alg_bytes": per_pass, "per": "one launch (one pass over U, P and W)",
                     "alg_bytes_note": "U and P rows + W + E rows + per-row inputs and "
                                       "partials; two launches per call, timed together",
                     "single_read_frac": achieved / 2 / peak},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches, "clocks": clk,
    }
    ctx.close()
    return line


def run_confidence(args, dsd, synth, dev, world):
    """The confidence side on the high-concurrency batch: the confidence head
    on R=256 requests x gamma positions (hidden size 2560, rank 256, V=151936;
    9.2 MB of hidden states, so L2 is flushed between steps outside the
    events), timed alone; calibration of 1M requests is timed beside it."""
    import torch

    R, G, H, V, r = 256, 7, 2560, 151936, 256
    x = synth.confidence_inputs(R, G, H, V, r, seed=7, dtype="bf16", device=dev)
    cal = synth.calibration_inputs(1 << 20, G, seed=8, device=dev)
    ctx = dsd.Context(V, r, G, R, dtype="bf16", device=dev.index)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    head_args = (x["h"], x["E"], x["w_c"], x["b_c"], x["prev_tok"], x["tokens"])
    out = cout = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            out = ctx.confidence_head(*head_args, out=out, stream=stream)
            cout = ctx.calibration(cal["conf"], cal["accept_len"], 10, out=cout, stream=stream)
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    c0 = ctx.launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(dev.index))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    with torch.cuda.stream(stream):
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            out = ctx.confidence_head(*head_args, out=out, stream=stream)
            e[1].record(stream)
            flush.zero_()
            e[2].record(stream)
            cout = ctx.calibration(cal["conf"], cal["accept_len"], 10, out=cout, stream=stream)
            e[3].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    assert ctx.sync_status(stream) == 0
    launches = ctx.launch_count() - c0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    cal_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    rows = R * G
    # per launch: every hidden row once, the Markov rows, w_c, tokens and outputs
    alg = rows * H * 2 + rows * r * 2 + (H + r) * 2 + rows * 4 + R * 4 + 2 * rows * 4
    cal_alg = (1 << 20) * G * 4 + (1 << 20) * 4
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": f"confidence-head rows/s (sigmoid(w_c . [h; E[t_prev]] + b_c) and survival) "
                  f"at R={R}, gamma={G}, H={H}, rank {r}",
        "value": world * rows / (ms / 1e3), "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "fp32 (fp64 survival)", "data": "synthetic",
        "config": {"workload": f"confidence: R={R} gamma={G} H={H} V={V} rank={r} bf16",
                   "l2": "flushed between steps (512 MB write outside the events); "
                         "inputs 9.2 MB"},
        "roofline": {"bound": "hbm", "kernel": "confidence_head_kernel", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": None, "alg_bytes": alg, "per": "one launch",
                     "alg_bytes_note": "hidden rows + Markov rows + w_c + tokens + outputs"},
        "calibration": {"requests": 1 << 20, "ms": cal_ms,
                        "achieved_gbs": cal_alg / (cal_ms / 1e3) / 1e9,
                        "frac": cal_alg / (cal_ms / 1e3) / 1e9 / peak},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches, "clocks": clk,
    }
    ctx.close()
    return line


def run_hidden_head(args, dsd, synth, dev, world, head):
    """A head that reads the backbone's hidden state -- the gated Markov head
    (head = "gated") or the RNN head ("rnn") -- proposing on the greedy
    workload (R=16 requests, gamma=7, V=151936, rank 256) with backbone
    hidden size 2560, on the --engine chosen (AUTO: the tensor-core engine's
    split mode; simt: the CUDA cores); L2 flushed between steps outside the
    events.  Beside it, the plain head's proposal on the same engine."""
    import torch

    spec = synth.CYCLE_SPECS["greedy"]
    H = 2560
    R, G, V, r = spec.R, spec.G, spec.V, spec.r
    x = synth.cycle_inputs(spec, device=dev)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine=args.engine,
                      device=dev.index)
    if head == "gated":
        hx = synth.gate_inputs(R, G, H, r, spec.ew_std, seed=66, device=dev)
        pa = (x["U"], x["E"], x["W"], hx["h"], hx["W_g"], x["conf"], x["prev_tok"])
        call = ctx.propose_gated
        weights = r * (H + r) * 2
        name, note = "gated-Markov-head", "W per step + U rows + h + W_g + E rows + gated reps"
    else:
        hx = synth.rnn_inputs(R, G, H, r, spec.ew_std, seed=67, device=dev)
        pa = (x["U"], x["E"], x["W"], hx["h"], hx["W_rnn"], x["conf"], x["prev_tok"])
        call = ctx.propose_rnn
        weights = 3 * r * (2 * r + H) * 2
        name, note = "RNN-head", "W per step + U rows + h + W_rnn + E rows + o_j"
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    out = plain = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            out = call(*pa, req_id=x["req_id"], out=out, stream=stream)
            plain = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                                req_id=x["req_id"], out=plain, stream=stream)
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    c0 = ctx.launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(dev.index))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    with torch.cuda.stream(stream):
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            out = call(*pa, req_id=x["req_id"], out=out, stream=stream)
            e[1].record(stream)
            flush.zero_()
            e[2].record(stream)
            plain = ctx.propose(x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                                req_id=x["req_id"], out=plain, stream=stream)
            e[3].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    assert ctx.sync_status(stream) == 0
    launches = ctx.launch_count() - c0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    plain_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    # per call: W every step (the CUDA-core engine re-reads it), every U row,
    # h and the head's weights once, the E rows, the representation written
    # and read
    alg = (G * V * r * 2 + R * G * V * 2 + R * G * H * 2 + weights + R * G * r * 2
           + 2 * R * G * r * 4)
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms / 1e3) / 1e9
    line = {
        "metric": f"{name} draft tokens/s at R=16, gamma=7, V=151936, rank 256, H=2560",
        "value": world * R * G / (ms / 1e3), "unit": "draft tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "fp32", "data": "synthetic",
        "config": {"workload": f"{head}: R={R} gamma={G} V={V} rank={r} H={H} bf16 greedy",
                   "l2": "flushed between steps (512 MB write outside the events); "
                         "inputs 0.6 GB per call"},
        "plain_head_ms": plain_ms,
        "engine": f"{args.engine} -> {ctx.last_engine()}",
        "roofline": {"bound": "hbm",
                     "kernel": ("propose_tc_kernel (split mode)" if ctx.last_engine() == "tcgen05"
                                else "simt_bias_kernel"),
                     "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": None, "alg_bytes": alg, "per": f"one {head} propose call",
                     "alg_bytes_note": note},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches, "clocks": clk,
    }
    if ctx.last_engine() == "simt":
        line["roofline"]["fma"] = fma_report(2.0 * R * r * V * G, ms / 1e3, "simt")
    ctx.close()
    return line


def run_gated(args, dsd, synth, dev, world):
    return run_hidden_head(args, dsd, synth, dev, world, "gated")


def run_rnn(args, dsd, synth, dev, world):
    return run_hidden_head(args, dsd, synth, dev, world, "rnn")


def run_candidates(args, dsd, synth, dev, world):
    """The proposal with the Markov top-16 candidate sets on the greedy
    workload (R=16, gamma=7, V=151936, rank 256) on the --engine chosen
    (AUTO: the tensor-core engine's repeated-rows kernel); beside it the
    plain proposal on the same engine; L2 flushed between steps."""
    import torch

    spec = synth.CYCLE_SPECS["greedy"]
    x = synth.cycle_inputs(spec, device=dev)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype="bf16", engine=args.engine,
                      device=dev.index)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    pa = (x["U"], x["E"], x["W"], x["conf"], x["prev_tok"])
    out = plain = None
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            out = ctx.propose_candidates(*pa, req_id=x["req_id"], out=out, stream=stream)
            plain = ctx.propose(*pa, req_id=x["req_id"], out=plain, stream=stream)
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    c0 = ctx.launch_count()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    clocks = ClockSampler(gpu_uuid(dev.index))
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    with torch.cuda.stream(stream):
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            out = ctx.propose_candidates(*pa, req_id=x["req_id"], out=out, stream=stream)
            e[1].record(stream)
            flush.zero_()
            e[2].record(stream)
            plain = ctx.propose(*pa, req_id=x["req_id"], out=plain, stream=stream)
            e[3].record(stream)
    stream.synchronize()
    clk = clocks.stop()
    assert ctx.sync_status(stream) == 0
    launches = ctx.launch_count() - c0
    ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    ms = max_over_ranks(ms, world, dev)
    plain_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    R, G, V, r = spec.R, spec.G, spec.V, spec.r
    alg = G * V * r * 2 + R * G * V * 2 + R * G * r * 2 + R * G * 16 * 8
    peak, peak_kind = hbm_peak()
    achieved = alg / (ms / 1e3) / 1e9
    eng = ctx.last_engine()
    line = {
        "metric": "draft tokens/s with Markov top-16 candidate sets at R=16, "
                  "gamma=7, V=151936, rank 256",
        "value": world * R * G / (ms / 1e3), "unit": "draft tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "accumulate": "fp32", "data": "synthetic",
        "config": {"workload": f"candidates: R={R} gamma={G} V={V} rank={r} bf16 greedy",
                   "l2": "flushed between steps (512 MB write outside the events)"},
        "plain_propose_ms": plain_ms,
        "engine": f"{args.engine} -> {eng}",
        "roofline": {"bound": "hbm",
                     "kernel": ("propose_tc_kernel (candidate mode)" if eng == "tcgen05"
                                else "simt_bias_kernel"),
                     "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                     "traffic": None, "alg_bytes": alg, "per": "one call",
                     "alg_bytes_note": "W per step + U rows + E rows + candidate sets"},
        "cpu_baseline": None, "e2e": None,
        "gpu_launches": launches, "clocks": clk,
    }
    if eng == "simt":
        line["roofline"]["fma"] = fma_report(2.0 * R * r * V * G, ms / 1e3, "simt")
    ctx.close()
    return line


def run_ours(args):
    import numpy as np
    import torch

    rank, local_rank, world = dist_info()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)

    import semi_autoregressive_draft_gb300 as dsd
    from semi_autoregressive_draft_gb300 import build as _build
    from semi_autoregressive_draft_gb300 import synth

    if not os.path.exists(dsd.LIB_PATH):
        _build.build()
    if args.workload in ("overlap", "loss", "confidence", "gated", "rnn", "candidates"):
        run = {"overlap": run_overlap, "loss": run_loss, "confidence": run_confidence,
               "gated": run_gated, "rnn": run_rnn, "candidates": run_candidates}[args.workload]
        line = run(args, dsd, synth, dev, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    spec = cycle_spec(args.workload)
    x = synth.cycle_inputs(spec, device=dev)
    ctx = dsd.Context(spec.V, spec.r, spec.G, spec.R, dtype=spec.dtype, engine=args.engine,
                      device=local_rank)
    T, seed = spec.temperature, x["seed"]
    out = ctx.cycle_outputs(spec.R)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)

    def propose():
        dsd.dsd_propose(ctx.handle, spec.R, x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                        x["req_id"], T, seed, out["tokens"], out["lse_q"], out["logit_at_tok"],
                        out["survival"], None, local_rank)

    def schedule():
        dsd.dsd_schedule(ctx.handle, spec.R, out["survival"], x["sps"], x["sps"].numel(),
                         out["keep_len"], out["theta_B"], None, local_rank)

    def verify():
        dsd.dsd_verify(ctx.handle, spec.R, x["P"], x["U"], x["E"], x["W"], x["prev_tok"],
                       out["tokens"], out["lse_q"], out["logit_at_tok"], out["keep_len"],
                       x["req_id"], T, seed, out["accept_len"], out["next_token"], None,
                       local_rank)

    def cycle():
        # the public one-call cycle: the schedule runs inside the proposal's
        # last launch
        dsd.dsd_cycle(ctx.handle, spec.R, x["U"], x["E"], x["W"], x["conf"], x["prev_tok"],
                      x["req_id"], x["P"], x["sps"], x["sps"].numel(), T, seed, out["tokens"],
                      out["lse_q"], out["logit_at_tok"], out["survival"], out["keep_len"],
                      out["theta_B"], out["accept_len"], out["next_token"], None, local_rank)

    with torch.cuda.stream(stream):
        for _ in range(2):               # eager warm-up (sets kernel attributes)
            propose(); schedule(); verify()
            cycle()
    stream.synchronize()
    assert ctx.sync_status(stream) == 0
    # the timed cycle is one graph; one graph per phase serves the breakdown
    g_cycle = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_cycle, stream=stream):
        cycle()
    # events recorded inside the propose and verify graphs (external event
    # nodes, where this torch has them) time each phase's launches without
    # the graph launch itself
    try:
        in_ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    except TypeError:
        in_ev = None
    graphs = []
    for k, fn in enumerate((propose, schedule, verify)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if in_ev and k != 1:
                in_ev[k // 2 * 2].record(stream)
            fn()
            if in_ev and k != 1:
                in_ev[k // 2 * 2 + 1].record(stream)
        graphs.append(g)
    launches_before_warm = ctx.launch_count()
    launches_per_cycle_eager = None

    def replay_cycle(ev=None):
        if ev:
            ev[0].record(stream)
        g_cycle.replay()
        if ev:
            ev[1].record(stream)

    def replay_phases(ev):
        for k in range(3):
            ev[k].record(stream)
            graphs[k].replay()
        ev[3].record(stream)

    # count kernels per cycle from the library's own launch counter
    c0 = ctx.launch_count()
    with torch.cuda.stream(stream):
        cycle()
    launches_per_cycle_eager = ctx.launch_count() - c0
    del launches_before_warm

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            replay_cycle()
    stream.synchronize()

    clocks = ClockSampler(gpu_uuid(local_rank)) if rank == 0 else None
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
        time.sleep(0.3)
    w0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            replay_cycle(evs[i])
    stream.synchronize()
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - w0
    clk = clocks.stop() if clocks else None
    st = ctx.sync_status(stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed region")

    cyc_ms = [e[0].elapsed_time(e[1]) for e in evs]

    # phase breakdown: the same cycles with one graph (and an event) per phase
    pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    prop_in, ver_in = [], []
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush.zero_()
            replay_phases(pevs[i])
            if in_ev:
                stream.synchronize()
                prop_in.append(in_ev[0].elapsed_time(in_ev[1]))
                ver_in.append(in_ev[2].elapsed_time(in_ev[3]))
    stream.synchronize()
    prop_ms = [e[0].elapsed_time(e[1]) for e in pevs]
    sch_ms = [e[1].elapsed_time(e[2]) for e in pevs]
    ver_ms = [e[2].elapsed_time(e[3]) for e in pevs]
    mean_cyc = statistics.mean(cyc_ms)
    mean_cyc_max = max_over_ranks(mean_cyc, world, dev)
    value = world * 1e3 / mean_cyc_max
    acc = out["accept_len"].cpu().numpy()
    keep = out["keep_len"].cpu().numpy()
    tokens_per_cycle = int((acc + 1).sum())
    B = int((keep + 1).sum())

    # the verify phase's read floor: where every request keeps the same
    # number of draft tokens, verification reads one row per request at the
    # same position; a library reduction over exactly those rows, captured
    # in a graph and timed like the verify phase, shows what a plain read of
    # those bytes costs on this GPU
    read_floor = None
    if (keep == keep[0]).all():
        rows = x["P"].view(spec.R, spec.G + 1, spec.V)[:, int(keep[0]), :]
        g_rf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rf, stream=stream):
            torch.amax(rows, dim=1)
        rf_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                  for _ in range(args.steps)]
        with torch.cuda.stream(stream):
            for ev in rf_evs:
                flush.zero_()
                ev[0].record(stream)
                g_rf.replay()
                ev[1].record(stream)
        stream.synchronize()
        rf_ms = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in rf_evs)
        rf_bytes = spec.R * spec.V * (2 if spec.dtype == "bf16" else 4)
        read_floor = {"kernel": "torch.amax over the rows verification reads (library kernel), "
                                "one graph per replay, L2 flushed before each",
                      "ms": rf_ms, "bytes": rf_bytes, "GBps": rf_bytes / (rf_ms / 1e3) / 1e9,
                      "verify_phase_ms": statistics.mean(ver_ms)}

    # acceptance of the scheduled cycle, and of one untimed pass that keeps
    # every draft position (l = gamma for all requests), so the histogram and
    # the per-position conditional accept rate cover every position
    keep_all = torch.full_like(out["keep_len"], spec.G)
    acc_all_t = torch.empty_like(out["accept_len"])
    nxt_all = torch.empty_like(out["next_token"])
    with torch.cuda.stream(stream):
        dsd.dsd_verify(ctx.handle, spec.R, x["P"], x["U"], x["E"], x["W"], x["prev_tok"],
                       out["tokens"], out["lse_q"], out["logit_at_tok"], keep_all,
                       x["req_id"], T, seed, acc_all_t, nxt_all, None, local_rank)
    stream.synchronize()
    acc_all = acc_all_t.cpu().numpy()
    acceptance = {
        "scheduled": {"accept_len_hist": np.bincount(acc, minlength=spec.G + 1).tolist(),
                      "keep_len_hist": np.bincount(keep, minlength=spec.G + 1).tolist(),
                      "mean_accept_len": float(acc.mean())},
        "keep_all": {"accept_len_hist": np.bincount(acc_all, minlength=spec.G + 1).tolist(),
                     "per_position_accept_rate": [
                         float((acc_all > i).sum() / max(1, (acc_all >= i).sum()))
                         for i in range(spec.G)],
                     "mean_accept_len": float(acc_all.mean())},
        "note": "per_position_accept_rate[i] = #(accept_len > i) / #(accept_len >= i), "
                "the rate at which position i is accepted once it is tested",
    }

    # e2e: same cycle from pinned host buffers through dsd_cycle_host
    e2e = None
    if not args.no_e2e:
        hU = x["U"].cpu().pin_memory()
        hP = x["P"].cpu().pin_memory()
        hc = x["conf"].cpu().pin_memory()
        hp = x["prev_tok"].cpu().pin_memory()
        hr = x["req_id"].cpu().pin_memory()
        ho = None
        for _ in range(max(1, min(args.warmup, 3))):
            ho = ctx.cycle_host(hU, x["E"], x["W"], hc, hp, hP, x["sps"], req_id_host=hr,
                                temperature=T, seed=seed, out=ho, stream=stream)
        n_e2e = max(3, min(args.steps, 10))
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            ho = ctx.cycle_host(hU, x["E"], x["W"], hc, hp, hP, x["sps"], req_id_host=hr,
                                temperature=T, seed=seed, out=ho, stream=stream)
        t_e2e = (time.perf_counter() - t0) / n_e2e
        t_e2e = max_over_ranks(t_e2e, world, dev)
        in_place = ctx.last_p_in_place()
        if in_place:
            # P read in place: the kept rows (and, sampled, each rejected row
            # once more for the residual) cross the CPU-GPU link
            row = spec.V * (2 if spec.dtype == "bf16" else 4)
            rejected = int((acc < keep).sum()) if T > 0 else 0
            p_bytes = (B + rejected) * row
        else:
            p_bytes = synth.bytes_of(hP)
        h2d = sum(synth.bytes_of(t) for t in (hU, hc, hp, hr)) + p_bytes
        d2h = sum(synth.bytes_of(ho[k]) for k in ("tokens", "keep_len", "accept_len", "next_token"))
        assert np.array_equal(ho["accept_len"].numpy(), acc)
        e2e = {"value": world / t_e2e, "unit": "cycles/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
               "path": "dsd_cycle_host (pinned host inputs; U staged by copy, P read in place "
                       "over the CPU-GPU link, only the kept rows)" if in_place else
                       "dsd_cycle_host (pinned host inputs, staging copies inside the call)"}

    peak, peak_kind = hbm_peak()
    pbytes = propose_alg_bytes(spec)
    # the propose phase's launches timed by the events inside its graph (the
    # phase without the graph launch); the phase pass's outer events where
    # this torch cannot record events inside a graph
    prop_mean_s = (statistics.mean(prop_in) if prop_in else statistics.mean(prop_ms)) / 1e3
    achieved = pbytes / prop_mean_s / 1e9
    w_once = propose_w_once_bytes(spec) / prop_mean_s / 1e9
    engine_used = ctx.last_engine()
    m_tiles = (spec.R + 127) // 128
    tc_kernel = "propose_tc_pair_kernel" if m_tiles >= 2 and m_tiles % 2 == 0 else "propose_tc_kernel"
    engine_kernel = {"tcgen05": tc_kernel, "mma": "propose_mma_kernel"}.get(
        engine_used, "simt_bias_kernel")
    roofline = {"bound": "hbm", "kernel": f"propose phase ({engine_kernel})",
                "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
                "traffic": traffic_for(engine_kernel, spec.name),
                "alg_bytes": propose_step_bytes(spec),
                "per": "one draft step (one launch covers all gamma steps); achieved = gamma "
                       "steps' bytes + the phase's small I/O over the propose call's mean time "
                       "(its memset, launch and finalize, timed by events inside the phase's "
                       "graph); traffic = DRAM bytes per draft step",
                "time_ms": prop_mean_s * 1e3,
                "time_kind": "events inside the propose graph" if prop_in else "phase events",
                "alg_bytes_note": "per step: the U rows of one position + all of W + the "
                                  "gathered E rows + the argmax keys",
                "w_once": {"achieved": w_once, "frac": w_once / peak,
                           "alg_bytes": propose_w_once_bytes(spec),
                           "note": "the same time against U rows once + W once per phase"},
                "tensor": tensor_report(spec, prop_mean_s, engine_used)}
    if engine_used == "simt":
        roofline["fma"] = fma_report(2.0 * spec.R * spec.r * spec.V * spec.G, prop_mean_s,
                                     engine_used)
    vbytes = verify_alg_bytes(spec, B)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = oracle_baseline(spec, x, n_cycles=args.cpu_cycles)

    line = {
        "metric": METRIC, "value": value, "unit": "cycles/s",
        "tokens_per_s": value * tokens_per_cycle, "tokens_per_cycle": tokens_per_cycle,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_cyc_max,
        "median_ms_per_step": statistics.median(cyc_ms),
        "wall_ms_per_step_incl_flush": wall * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": spec.dtype, "accumulate": "fp32", "data": "synthetic",
        "config": cycle_config(spec, world),
        "engine": f"{args.engine} -> {engine_used}", "verify_batch_B": B,
        "phases_ms": {"propose": statistics.mean(prop_ms), "schedule": statistics.mean(sch_ms),
                      "verify": statistics.mean(ver_ms),
                      "note": "separate pass through dsd_propose, dsd_schedule and dsd_verify, "
                              "one graph each (adds a graph launch each); the timed cycle "
                              "(dsd_cycle) runs the schedule inside the proposal's last launch"},
        "verify_alg_GBps": vbytes / (statistics.mean(ver_ms) / 1e3) / 1e9,
        "phases_in_graph_ms": ({"propose": statistics.mean(prop_in),
                                "verify": statistics.mean(ver_in),
                                "verify_alg_GBps": vbytes / (statistics.mean(ver_in) / 1e3) / 1e9,
                                "note": "events recorded inside each phase's graph around the "
                                        "call's launches: the phase without the graph launch"}
                               if prop_in else None),
        "verify_read_floor": read_floor,
        "acceptance": acceptance,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(launches_per_cycle_eager * args.steps),
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="highconc",
                    choices=["highconc", "greedy", "sampled", "tiny", "overlap", "loss",
                             "confidence", "gated", "rnn", "candidates"])
    ap.add_argument("--engine", default="auto", choices=["auto", "simt", "mma", "tcgen05"])
    ap.add_argument("--cpu-cycles", type=int, default=2,
                    help="timed full-batch oracle cycles of the in-run CPU baseline")
    ap.add_argument("--ref-requests", type=int, default=0,
                    help="reference arm: requests proposed and verified per step (default 0: "
                         "the whole batch)")
    ap.add_argument("--blocks", type=int, default=0,
                    help="overlap workload: blocks N instead of 4096 (small profiling cases)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least 3 untimed warm-up steps
    if args.impl == "reference":
        if args.workload in ("overlap", "loss", "confidence", "gated", "rnn", "candidates"):
            ap.error("the reference arm times the draft-verify cycle workloads")
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
