#!/usr/bin/env python3
"""Benchmark of the B300 Entropy-Bounded (EB) sampler step of DiffusionGemma.

One step = the whole hot path over one canvas batch: temperature shaping, per-position
softmax entropy / argmax / Gumbel-max sample over the full vocabulary, entropy-bounded
selection, re-mask and stop test (DiffusionGemma model card, "Best practices" section 1).
Workload: B=1 canvas, L=256 positions, V=262144 bf16 logits = 2.5 N(0,1) plus a U(0,12)
peak per position, 128 of 256 positions masked, T=0.8; ten seeded logit buffers (seeds
0..9, 10 x 128 MiB > the 126 MB L2) are rotated, and every step starts from a fresh copy
of its canvas state so each step does the same work.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun (N > 1) every rank runs its own replica
(the sampler has no cross-canvas exchange) and the value is all ranks' steps over the
slowest rank's time.  ``--impl reference`` times the CPU oracle on the host cores instead.

The headline line also carries, under "workloads", one record per other workload, each
measured in the same run on the same GPU: the fused unembedding step (4 canvases and one),
the full adaptive loop of one canvas and of the mixed batch of eight (steps to stop, tokens
committed per step), the e4m3 single step and the block driver.  ``--workload NAME`` prints
one of them as the line instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "EB-sampler steps/s at B×256×262144 bf16; achieved HBM GB/s vs B300 peak"
B, L, V = 1, 256, 262144
NSEEDS = 10
K1_SAMPLES = 100                         # row-statistics launches timed one by one
WARM_SECONDS = 0.5                       # least time of warm-up steps before any timed work
BYTES_PER_STEP = B * L * V * 2           # algorithmic bytes: every logit read once
TEMPERATURE = 0.8
FLUSH_ELEMS = 1 << 29                # int16 elements (1 GiB) written right before a timed region
WORKLOAD = ("single EB sampler step: B=1 canvas, L=256 positions, V=262144 bf16 logits "
            "(2.5*N(0,1) + U(0,12) peak per position), 128 of 256 masked, T=0.8")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k1_rowstats_bf16_single_step.md")
KERNEL_SRCS = [os.path.join(ROOT, "canvas_sampler_step_b300", "csrc", f)
               for f in ("eb_sampler.cu", "eb_kernels.cuh")]


def _strip_comments(text: str) -> str:
    """C++ source without // and /* */ comments or trailing blanks (string literals in these
    sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the row-statistics kernel's sources, comments
    left out, so that a comment edit does not void a recorded traffic figure."""
    h = hashlib.sha256()
    for f in KERNEL_SRCS:
        with open(f, encoding="utf-8") as fh:
            h.update(_strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--logits", choices=("bf16", "fp8"), default="bf16",
                    help="element type of the single-step workload's logits (fp8: OCP e4m3)")
    ap.add_argument("--workload", choices=("single", "fused", "fused1", "loop", "loop1", "stop", "blocks"),
                    default="single",
                    help="single: the single-step workload (default, the headline line); fused: "
                         "the fused unembedding + sampler step (4 x 256 positions, K=2048); "
                         "fused1: the same for one canvas (256 positions); loop: the adaptive "
                         "48-step loop over 8 canvases with the stand-in denoiser; loop1: the "
                         "same for one canvas; stop: a one-canvas loop that the adaptive stop "
                         "ends early; blocks: the block driver, 64 blocks on 8 slots")
    ap.add_argument("--no-extras", action="store_true",
                    help="headline only: leave out the per-workload records")
    return ap.parse_args(argv)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device=None) -> float:
    """Maximum of a per-rank scalar (timing) over all ranks."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64,
                     device=f"cuda:{device}" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(steps_per_rank: int, elapsed_s: float, world: int, dist=None, device=None):
    """(whole-job steps/s, slowest rank's seconds): steps of all ranks / max time."""
    slowest = max_over_ranks(dist, elapsed_s, device)
    return steps_per_rank * world / slowest, slowest


# ------------------------------------------------------------------ peaks, traffic, clocks

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def recorded_traffic():
    """Per-launch DRAM bytes of the row-statistics kernel from the committed ncu summary,
    or None when absent or taken on a different kernel source."""
    try:
        text = open(TRAFFIC_FILE).read()
        src_hash = kernel_source_hash()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line and line.startswith(("traffic_bytes_per_launch", "kernel_source_sha256")):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != src_hash:
        return None
    try:
        return int(float(vals["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """Samples SM clock, power and clock-event reasons with nvidia-smi (200 ms period) while
    the timed region runs."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMED = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, log_path: str | None = None):
        import tempfile
        self.device_index = device_index
        self.log_path = log_path or tempfile.mktemp(prefix="eb_clocks_", suffix=".csv")
        self.proc = None
        self.rows = []

    def _target(self):
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.device_index)
            return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            return str(self.device_index)

    def __enter__(self):
        import subprocess
        try:
            self._f = open(self.log_path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self._target(), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self._f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        self.t0 = time.time()
        return self

    def __exit__(self, *exc):
        self.t1 = time.time()
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self._f.close()
            import datetime
            for line in open(self.log_path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except ValueError:
                    ts = None
                # keep the samples taken while the timed region ran (one period of slack)
                if ts is None or self.t0 - 0.2 <= ts <= self.t1 + 0.2:
                    self.rows.append(f)

    def summary(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        mhz = [num(r[1]) for r in self.rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in self.rows if num(r[2]) is not None]
        reasons = set()
        for r in self.rows:
            for name, val in zip(self.NAMED, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(self.rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in self.rows) if self.rows else None}


# ------------------------------------------------------------------ the workload

def logits_kind(args, eb, torch):
    """Element type of the single-step workload: bf16 (the headline) or OCP e4m3."""
    import dataclasses

    import eb_synth
    if getattr(args, "logits", "bf16") == "fp8":
        return {"name": "e4m3", "torch": torch.uint8, "eb": eb.EB_FP8_E4M3, "bytes": B * L * V,
                "cfg": lambda seed: dataclasses.replace(eb_synth.cfg1(seed), dtype="fp8"),
                "metric": METRIC.replace("bf16", "e4m3"),
                "workload": WORKLOAD.replace("bf16 logits", "e4m3 logits (the bf16 workload's values "
                                             "rounded to e4m3)")}
    return {"name": "bf16", "torch": torch.int16, "eb": eb.EB_BF16, "bytes": BYTES_PER_STEP,
            "cfg": eb_synth.cfg1, "metric": METRIC, "workload": WORKLOAD}


def workload_masks():
    import eb_synth
    return np.stack([eb_synth.cfg1_mask(seed)[0] for seed in range(NSEEDS)])


def state_pool(n: int, masks: np.ndarray, device):
    """n fresh canvas states; state i belongs to logits buffer i % NSEEDS."""
    import torch
    idx = np.arange(n) % NSEEDS
    m = torch.from_numpy(masks[idx]).to(device)
    pool = {
        "mask": m,
        "tokens": torch.where(m.bool(), -1, 0).to(torch.int32),
        "prev_argmax": torch.full((n, L), -1, dtype=torch.int32, device=device),
        "status": torch.zeros(n, dtype=torch.int32, device=device),
        "steps_taken": torch.zeros(n, dtype=torch.int32, device=device),
        "entropy": torch.zeros((n, L), dtype=torch.float32, device=device),
        "argmax": torch.zeros((n, L), dtype=torch.int32, device=device),
        "sampled": torch.zeros((n, L), dtype=torch.int32, device=device),
        "selected": torch.zeros((n, L), dtype=torch.uint8, device=device),
        "committed": torch.zeros(n, dtype=torch.int32, device=device),
        "mean_entropy": torch.zeros(n, dtype=torch.float32, device=device),
    }
    return pool


_ORDER = ("mask", "tokens", "prev_argmax", "status", "steps_taken", "entropy", "argmax",
          "sampled", "selected", "committed", "mean_entropy")


def state_ptrs(pool, i):
    out = []
    for k in _ORDER:
        t = pool[k]
        row = t[i] if t.dim() > 1 else t[i:i + 1]
        out.append(row.data_ptr())
    return out


def k1_graph_samples(lib, one, masks, device, torch, steps=20, replays=5):
    """CUDA-event durations (ms) of steps x replays row-statistics launches: a CUDA graph of
    `steps` whole steps (after a restore of their canvas states), each with its row-statistics
    launch between its own pair of events (eb_set_profile_events during capture), replayed
    `replays` times; the durations are read after every replay."""
    pool = state_pool(steps, masks, device)
    pristine = {k: v.clone() for k, v in pool.items()}
    ptrs = [state_ptrs(pool, i) for i in range(steps)]
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    stream = torch.cuda.current_stream(device)
    for b, e in evs:
        b.record(stream)
        e.record(stream)          # materialise the CUDA events before capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        graph.capture_begin()
        for k in pool:
            pool[k].copy_(pristine[k])
        csp = torch.cuda.current_stream(device).cuda_stream
        for j, (b, e) in enumerate(evs):
            lib.eb_set_profile_events(b.cuda_event, e.cuda_event)
            one(j, ptrs, csp)
        graph.capture_end()
    torch.cuda.synchronize()
    graph.replay()                # untimed
    torch.cuda.synchronize()
    ms = []
    for _ in range(replays):
        graph.replay()
        torch.cuda.synchronize()
        ms += [b.elapsed_time(e) for b, e in evs]
    return ms


def sample_stats(ms):
    """median / p10 / p90 / mean of a list of durations (ms), and their count."""
    a = np.sort(np.asarray(ms, dtype=np.float64))
    return {"n": int(a.size), "median_ms": float(np.median(a)), "p10_ms": float(np.percentile(a, 10)),
            "p90_ms": float(np.percentile(a, 90)), "mean_ms": float(a.mean())}


def single_step_setup(args, lk, device, W):
    """Resident inputs of the single-step workload: NSEEDS rotating logit buffers, the initial
    masks, a pool of W canvas states and the workspace."""
    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth.device as synth_dev
    bufs = []
    for seed in range(NSEEDS):
        x = torch.empty((B, L, V), dtype=lk["torch"], device=device)
        synth_dev.logits(synth_dev.Recipe.of(lk["cfg"](seed)), 0, x)
        bufs.append(x)
    masks = workload_masks()
    ws_bytes = eb.eb_workspace_bytes(B, L, V, lk["eb"])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    return bufs, masks, ws, ws_bytes


def run_single(args, lk, device, local, dist, world, timed=True):
    """The single-step workload (bf16 or e4m3 logits): the timed region is `steps` steps as
    replays of a CUDA graph of N steps (with a canvas-state restore before every replay but the
    first, which runs before the timed region), then K1_SAMPLES row-statistics launches timed
    one by one.  Returns the measurement dict."""
    import ctypes

    import torch

    import canvas_sampler_step_b300 as eb
    lib = eb.lib()
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream
    K, W = args.steps, max(args.warmup, 3)
    bufs, masks, ws, ws_bytes = single_step_setup(args, lk, device, W)
    # the timed steps run as replays of a CUDA graph of N steps (N divides K), so the host's
    # per-call cost stays out of the device time; its N canvas states are restored from a
    # pristine copy before each replay, so every step does the workload's work
    N = max(d for d in range(1, min(K, 200) + 1) if K % d == 0)
    R = K // N
    pool = state_pool(N, masks, device)
    pristine = {k: v.clone() for k, v in pool.items()}
    ptrs = [state_ptrs(pool, i) for i in range(N)]
    wpool = state_pool(W, masks, device)
    wptrs = [state_ptrs(wpool, i) for i in range(W)]
    params = eb.eb_default_params(seed=0)
    pref = ctypes.byref(params)
    buf_ptrs = [b.data_ptr() for b in bufs]
    wsp = ws.data_ptr()
    step_fn = lib.eb_sampler_step

    def one(i, sptrs, stream_ptr):
        st = step_fn(pref, B, L, V, lk["eb"], buf_ptrs[i % NSEEDS], 0, TEMPERATURE, *sptrs[i % len(sptrs)],
                     wsp, ws_bytes, stream_ptr)
        if st != 0:
            raise eb.EbError(st, lib.eb_last_error().decode())

    for i in range(W):
        one(i, wptrs, sp)
    torch.cuda.synchronize()
    # two graphs: the canvas-state restore, and the N steps
    restore = torch.cuda.CUDAGraph()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        restore.capture_begin()
        for k in pool:
            pool[k].copy_(pristine[k])
        restore.capture_end()
        graph.capture_begin()
        csp = torch.cuda.current_stream(device).cuda_stream
        for j in range(N):
            one(j, ptrs, csp)
        graph.capture_end()
    torch.cuda.synchronize()
    # warm-up by time as well as by count: the GPU runs this kernel several per cent slower for
    # the first few hundred launches of a process, so the graph is replayed for WARM_SECONDS
    # (at least once) before anything is timed
    warm_replays = 0
    t0 = time.perf_counter()
    while warm_replays < 1 or time.perf_counter() - t0 < WARM_SECONDS:
        restore.replay()
        graph.replay()
        torch.cuda.synchronize()
        warm_replays += 1
    # the canvas states start pristine; a restore between replays (K > N) stays in the timed
    # region, so that every timed step does the workload's work
    restore.replay()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dist, local)
    torch.cuda.synchronize()
    flush = torch.empty(FLUSH_ELEMS, dtype=torch.int16, device=device)
    with ClockSampler(local) as clocks:
        # writing 1 GiB (far more than L2) right before the start event flushes L2 and keeps the
        # GPU and its memory busy while the host queues the replays, so that the host's graph
        # submission stays out of the device time
        flush.fill_(1)
        start.record(stream)
        for r in range(R):
            if r > 0:
                restore.replay()
            graph.replay()
        end.record(stream)
        torch.cuda.synchronize()
    barrier(dist, local)
    del flush
    elapsed = start.elapsed_time(end) / 1e3
    value, slowest = aggregate(K, elapsed, world, dist, local)
    # every timed step did the workload's work: running canvas, one position committed
    st = pool["status"].cpu().numpy()
    com = pool["committed"].cpu().numpy()
    if not ((st == 0).all() and (com >= 1).all()):
        raise RuntimeError("timed steps did not run the expected workload")

    # the row-statistics kernel alone: K1_SAMPLES launches inside replays of a timing graph,
    # each between its own events
    k1_ms = k1_graph_samples(lib, one, masks, device, torch, steps=20, replays=K1_SAMPLES // 20)
    k1 = sample_stats(k1_ms)
    return {"value": value, "elapsed": elapsed, "slowest": slowest, "K": K, "W": W, "N": N, "R": R,
            "k1": k1, "clocks": clocks.summary(), "bufs": bufs, "masks": masks, "params": params,
            "stream": stream, "warm_steps": W + warm_replays * N}


def run_ours(args, rank, world, local):
    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth.device as synth_dev

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    lib = eb.lib()
    synth_dev.lib()
    lk = logits_kind(args, eb, torch)
    m = run_single(args, lk, device, local, dist, world)
    K, W = m["K"], m["W"]
    peak, peak_kind = measured_peaks()
    k1 = m["k1"]
    achieved = lk["bytes"] / (k1["median_ms"] / 1e3) / 1e9
    traffic = recorded_traffic() if lk["name"] == "bf16" else None
    e2e = run_e2e(args, eb, lib, m["bufs"], m["masks"], m["params"], device, m["stream"], dist, local, world, lk)
    out = {
        "metric": lk["metric"],
        "value": m["value"],
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": m["slowest"] * 1e3 / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded Philox / Box-Muller logits, eb_synth)",
        "config": {
            "workload": lk["workload"],
            "B": B, "L": L, "V": V, "logits_dtype": lk["name"], "masked": 128, "temperature": TEMPERATURE,
            "l2": f"10 rotating {lk['bytes'] >> 20} MiB logit buffers ({10 * lk['bytes'] / 2**30:.3g} GiB > 126 MB L2), "
                  "and a 1 GiB write right before the timed region",
            "launch": f"CUDA graph of {m['N']} steps replayed {m['R']} times (canvas states restored before "
                      "each replay, in the timed region from the second on) "
                      f"after {m['warm_steps']} warm-up steps (at least {WARM_SECONDS} s); row-statistics "
                      f"kernel timed separately over {K1_SAMPLES} launches: a second graph of 20 steps with "
                      "CUDA events around each row-statistics launch, replayed "
                      f"{K1_SAMPLES // 20} times",
            "parallelism": f"replicas x{world}",
        },
        "hbm_gbs_step": lk["bytes"] * K / m["elapsed"] / 1e9,
        "positions_per_s": m["value"] * B * L,
        "roofline": {
            "bound": "hbm",
            "kernel": f"k1_rowstats<{lk['name']}>",
            "achieved": achieved,
            "peak": peak,
            "peak_kind": f"{peak_kind} (copy, MEASURED_PEAKS hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": traffic,
            "traffic_source": (f"recorded: ncu dram__bytes_read.sum + dram__bytes_write.sum per launch, from "
                               f"profiles/k1_rowstats_bf16_single_step.md, taken on kernel sources with hash "
                               f"{kernel_source_hash()} (the sources of this run)") if traffic is not None
                              else "none recorded for these kernel sources",
            "k1_ms_median": k1["median_ms"],
            "k1_ms_p10": k1["p10_ms"],
            "k1_ms_p90": k1["p90_ms"],
            "k1_ms_mean": k1["mean_ms"],
            "k1_samples": k1["n"],
            "bytes_per_launch": lk["bytes"],
        },
        "e2e": e2e,
        "gpu_launches": 2 * K,                 # row statistics + selection per step
        "clocks": m["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_extras and lk["name"] == "bf16":
        out["workloads"] = extras(args, device, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, eb, lib, bufs, masks, params, device, stream, dist, local, world, lk):
    """Same steps through the C ABI with host buffers: per step the pinned-host logits
    and canvas state go to the device, the step runs, its results come back."""
    import ctypes

    import torch
    n = max(1, min(args.e2e_steps, args.steps))
    host_logits = [b.cpu().pin_memory() for b in bufs]
    dev_logits = torch.empty_like(bufs[0])
    in_keys = ("mask", "tokens", "prev_argmax", "status")
    hpool = state_pool(NSEEDS, masks, "cpu")
    hstate = [{k: hpool[k][s:s + 1].clone().pin_memory() for k in in_keys} for s in range(NSEEDS)]
    dstate = state_pool(1, masks, device)
    ptrs = state_ptrs(dstate, 0)
    out_keys = ("tokens", "mask", "status", "entropy", "argmax", "sampled", "selected")
    hout = {k: torch.empty_like(dstate[k], device="cpu").pin_memory() for k in out_keys}
    ws_bytes = eb.eb_workspace_bytes(B, L, V, lk["eb"])
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    pref = ctypes.byref(params)
    sp = stream.cuda_stream
    h2d = host_logits[0].numel() * host_logits[0].element_size() + sum(
        hstate[0][k].numel() * hstate[0][k].element_size() for k in in_keys)
    d2h = sum(hout[k].numel() * hout[k].element_size() for k in out_keys)

    def one(i):
        s = i % NSEEDS
        dev_logits.copy_(host_logits[s], non_blocking=True)
        for k in in_keys:
            dstate[k].copy_(hstate[s][k], non_blocking=True)
        st = lib.eb_sampler_step(pref, B, L, V, lk["eb"], dev_logits.data_ptr(), 0, TEMPERATURE,
                                 *ptrs, ws.data_ptr(), ws_bytes, sp)
        if st != 0:
            raise eb.EbError(st, lib.eb_last_error().decode())
        for k in out_keys:
            hout[k].copy_(dstate[k], non_blocking=True)

    for i in range(3):
        one(i)
    torch.cuda.synchronize()
    barrier(dist, local)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(n):
        one(i)
    end.record(stream)
    torch.cuda.synchronize()
    elapsed = start.elapsed_time(end) / 1e3
    value, _ = aggregate(n, elapsed, world, dist, local)
    return {"value": value, "unit": "steps/s", "steps": n, "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------------------ CPU oracle legs

def cpu_baseline():
    """The oracle, as it stands, on full steps of the workload (seed 0: 256 rows x 262144
    bf16, 128 masked): the median of three steps with all its OpenMP threads on the host
    cores, and one step on a single thread."""
    import eb_synth
    import oracle
    cfg = eb_synth.cfg1(0)
    x = cfg.logits(0)
    mask = eb_synth.cfg1_mask(0)

    def one():
        st = oracle.State.fresh(B, L, mask)
        t0 = time.perf_counter()
        oracle.step(x, st, 0, oracle.Params(seed=0), temperature=float(np.float32(TEMPERATURE)))
        return time.perf_counter() - t0

    cores = oracle.num_threads()
    dt = statistics.median(one() for _ in range(3))
    oracle.set_num_threads(1)
    try:
        dt1 = one()
    finally:
        oracle.set_num_threads(cores)
    return {"value": 1.0 / dt, "unit": "steps/s", "cores": cores, "kind": "oracle",
            "one_thread_value": 1.0 / dt1,
            "sample": "full steps of seed 0 (256 rows x 262144 bf16, 128 masked), all rows and the "
                      f"selection: median of 3 on {cores} threads ({dt:.2f} s wall each), "
                      f"1 on one thread ({dt1:.2f} s)",
            "parity": step_parity(x, mask)}


def step_parity(x, mask):
    """The library's step next to the oracle's on the same input (seed 0 of the workload),
    with the near-ties counted as the parity tests count them: entropy error, argmax and
    sample mismatches, and whether the selection matched."""
    import torch

    import canvas_sampler_step_b300 as eb
    import oracle
    st = oracle.State.fresh(B, L, mask)
    res = oracle.step(x, st, 0, oracle.Params(seed=0), temperature=float(np.float32(TEMPERATURE)))
    c = eb.Canvas(B, L, V, eb.EB_BF16, mask=mask)
    c.step(eb.eb_default_params(seed=0), torch.from_numpy(x.view(np.int16)).cuda(), 0, TEMPERATURE)
    torch.cuda.synchronize()
    return parity_summary(c.entropy.cpu().numpy().astype(np.float64), c.argmax.cpu().numpy(),
                          c.sampled.cpu().numpy(), c.mask.cpu().numpy(), mask, res, st.mask)


def parity_summary(H, A, Y, mask_after, mask_before, res, oracle_mask_after):
    """The step's agreement with the oracle's result ``res``: the largest entropy error, argmax
    mismatches, sample mismatches of masked rows apart from near-ties (top-2 perturbed-score gap
    below 1e-6), those near-ties, whether the selection left the same mask, and whether the
    selection itself was a near-tie (a prefix sum within 1e-5 of the bound, or an acceptance cut
    between entropies closer than 2e-5)."""
    masked = mask_before.astype(bool)
    ydiff = masked & (Y != res.Y)
    ties = res.gap < 1e-6
    canvas_tie = bool((res.sum_margin <= 1e-5).any() or (res.order_margin <= 2e-5).any())
    return {"rows": int(H.size), "max_abs_dH": float(np.abs(H - res.H).max()),
            "argmax_mismatch": int((A != res.A).sum()),
            "sample_mismatch": int((ydiff & ~ties).sum()), "sample_ties": int((ydiff & ties).sum()),
            "selection_equal": bool(np.array_equal(mask_after, oracle_mask_after)),
            "canvas_tie": canvas_tie}


def run_reference(args, rank, world, local):
    """The oracle as the reference arm: every step is a bounded sample of the workload
    (R rows of n logits from seed 0, half of them masked), timed on the host cores and
    scaled to full steps by the element count."""
    if rank != 0:
        return
    import eb_synth
    import oracle
    K, W = args.steps, args.warmup
    R = 64
    cfg = eb_synth.cfg1(0)
    masks = eb_synth.cfg1_mask(0)[0]
    rows = np.concatenate([np.nonzero(masks)[0][:R // 2], np.nonzero(masks == 0)[0][:R // 2]])
    full = cfg.rows(0, rows, 0)                     # [R, V]
    params = oracle.Params(seed=0)
    T = float(np.float32(TEMPERATURE))
    sub_mask = masks[rows][None, :]

    def run(n):
        x = np.ascontiguousarray(full[None, :, :n])
        st = oracle.State.fresh(1, R, sub_mask)
        t0 = time.perf_counter()
        oracle.step(x, st, 0, params, temperature=T)
        return time.perf_counter() - t0

    # size the sample so that K + W steps take about two minutes at most
    t_full = run(V)
    budget = 120.0
    n = V
    if t_full * (K + W) > budget:
        n = max(1024, int(V * budget / (t_full * (K + W))) // 8 * 8)
    for _ in range(W):
        run(n)
    times = [run(n) for _ in range(K)]
    elapsed = sum(times)
    elems_per_step = R * n
    value = K * elems_per_step / (B * L * V) / elapsed
    out = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "steps/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": 1e3 / value,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded Philox / Box-Muller logits, eb_synth)",
        "config": {"workload": WORKLOAD, "B": B, "L": L, "V": V, "logits_dtype": "bf16",
                   "masked": 128, "temperature": TEMPERATURE,
                   "l2": "host cores, not applicable", "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": oracle.num_threads(),
                         "kind": "oracle",
                         "sample": f"each step: oracle on {R} rows ({R // 2} masked) x {n} logits "
                                   f"of seed 0, scaled by {B * L * V}/{elems_per_step} elements"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ fused unembedding workload

FUSED_METRIC = ("EB-sampler fused unembedding steps/s at {B}x256 positions, K=2048, V=262144 bf16; "
                "achieved tensor TFLOP/s vs B300 peak")
FL, FK, FV = 256, 2048, 262144


def measured_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 1400.0, 1800.0, "fallback"


def measure_fused(FB, K, Wm, e2e_steps, device, local, dist=None, world=1):
    """One step = eb_unembed_sample over FB x 256 fresh all-masked positions: h [256 FB, 2048]
    x W [2048, 262144] on the tensor cores, the row statistics in the epilogue, the selection.
    h and W are resident (W is the model's unembedding matrix); each graph replay restores the
    canvas states first.  Returns the measurement dict (the line's fields)."""
    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth.device as synth_dev

    FUSED_FLOP = 2 * FB * FL * FK * FV
    lib = eb.lib()
    stream = torch.cuda.current_stream(device)
    h = torch.empty((FB * FL, FK), dtype=torch.int16, device=device)
    W = torch.empty((FK, FV), dtype=torch.int16, device=device)
    synth_dev.unembed_inputs(0, FB * FL, FK, FV, 0.02, 0.05, h, W)
    N = max(d for d in range(1, min(K, 20) + 1) if K % d == 0)
    R = K // N
    canv = [eb.Canvas(FB, FL, FV, eb.EB_BF16, device=device) for _ in range(N)]
    pristine = {k: getattr(canv[0], k).clone() for k in ("mask", "tokens", "prev_argmax", "status",
                                                          "steps_taken")}
    ws_bytes = eb.eb_unembed_workspace_bytes(FB, FL, FK, FV)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    params = eb.eb_default_params(seed=0)

    def one(c, sp):
        eb.eb_unembed_sample(params, FB, FL, FK, FV, h, W, 0, 0.8, c.mask, c.tokens, c.prev_argmax,
                             c.status, c.steps_taken, c.entropy, c.argmax, c.sampled, c.selected,
                             c.committed, c.mean_entropy, ws, ws_bytes, sp)

    warm = eb.Canvas(FB, FL, FV, eb.EB_BF16, device=device)
    for _ in range(max(Wm, 3)):
        for k, v in pristine.items():
            getattr(warm, k).copy_(v)
        one(warm, stream.cuda_stream)
    torch.cuda.synchronize()
    kb = [torch.cuda.Event(enable_timing=True) for _ in range(N)]
    ke = [torch.cuda.Event(enable_timing=True) for _ in range(N)]   # ~1 ms steps: 8 us is noise
    for e in kb + ke:
        e.record(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(device)
    with torch.cuda.stream(cap):
        graph.capture_begin()
        csp = torch.cuda.current_stream(device).cuda_stream
        for j in range(N):
            for k, v in pristine.items():
                getattr(canv[j], k).copy_(v)
            lib.eb_set_profile_events(kb[j].cuda_event, ke[j].cuda_event)
            one(canv[j], csp)
        graph.capture_end()
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier(dist, local)
    k3_ms = []
    with ClockSampler(local) as clocks:
        start.record(stream)
        for _ in range(R):
            graph.replay()
            k3_ms += [b.elapsed_time(e) for b, e in zip(kb, ke)] if False else []
        end.record(stream)
        torch.cuda.synchronize()
    barrier(dist, local)
    elapsed = start.elapsed_time(end) / 1e3
    k3_ms = [b.elapsed_time(e) for b, e in zip(kb, ke)]          # the last replay's steps
    value, slowest = aggregate(K, elapsed, world, dist, local)
    for c in canv:
        if not ((c.status == 0).all() and (c.committed >= 1).all()):
            raise RuntimeError("timed steps did not run the expected workload")
    sustained, burst, kind = measured_tensor_peak()
    k3 = sample_stats(k3_ms)
    achieved = FUSED_FLOP / (k3["median_ms"] / 1e3) / 1e12

    # end to end: per step the hidden states and canvas state go host -> device, the step
    # runs, the results come back (W stays resident: it is the model's weight)
    n_e2e = max(1, min(e2e_steps, 50))
    h_host = h.cpu().pin_memory()
    in_keys = ("mask", "tokens", "prev_argmax", "status")
    hstate = {k: pristine[k].cpu().pin_memory() for k in in_keys}
    out_keys = ("tokens", "mask", "status", "entropy", "argmax", "sampled", "selected")
    c = canv[0]
    hout = {k: torch.empty_like(getattr(c, k), device="cpu").pin_memory() for k in out_keys}
    h_dev = torch.empty_like(h)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n_e2e):
        h_dev.copy_(h_host, non_blocking=True)
        for k in in_keys:
            getattr(c, k).copy_(hstate[k], non_blocking=True)
        eb.eb_unembed_sample(params, FB, FL, FK, FV, h_dev, W, 0, 0.8, c.mask, c.tokens,
                             c.prev_argmax, c.status, c.steps_taken, c.entropy, c.argmax,
                             c.sampled, c.selected, c.committed, c.mean_entropy, ws, ws_bytes,
                             stream.cuda_stream)
        for k in out_keys:
            hout[k].copy_(getattr(c, k), non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(n_e2e, e0.elapsed_time(e1) / 1e3, world, dist, local)
    h2d = h_host.numel() * 2 + sum(v.numel() * v.element_size() for v in hstate.values())
    d2h = sum(v.numel() * v.element_size() for v in hout.values())
    del W, h, h_dev
    return {
        "metric": FUSED_METRIC.format(B=FB), "value": value, "unit": "steps/s", "steps": K,
        "warmup": Wm, "ms_per_step": slowest * 1e3 / K, "higher_is_better": True, "dtype": "bf16",
        "config": {"workload": f"fused unembedding + EB sampler step: h [{FB * FL}, 2048] ~ N(0,1) x W "
                               "[2048, 262144] ~ N(0, 0.02^2) + 0.05 planted per row, bf16, "
                               f"{FB} canvas{'es' if FB > 1 else ''} x 256 positions all masked, T=0.8",
                   "B": FB, "L": FL, "K": FK, "V": FV,
                   "l2": "W (1 GiB) > 126 MB L2, read once per step",
                   "launch": f"CUDA graph of {N} steps (+ canvas-state restores) replayed {R} times; "
                             "the fused kernel timed by events around each step of the last replay"},
        "roofline": {"bound": "tensor", "kernel": "k3_unembed", "achieved": achieved,
                     "peak": sustained, "unit": "TFLOP/s", "frac": achieved / sustained,
                     "peak_kind": f"{kind} bf16 sustained (burst {burst})", "traffic": None,
                     "k3_ms_median": k3["median_ms"], "k3_ms_p10": k3["p10_ms"], "k3_ms_p90": k3["p90_ms"],
                     "k3_samples": k3["n"], "flop_per_launch": FUSED_FLOP},
        "e2e": {"value": e2e_value, "unit": "steps/s", "steps": n_e2e, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": 2 * K,
        "clocks": clocks.summary(),
    }


# ------------------------------------------------------------------ block driver workload

BLOCKS_METRIC = ("EB block driver (continuous batching): blocks/s over 64 blocks x 256 x 262144 bf16 "
                 "on 8 slots, stand-in denoiser included")


def measure_blocks(device, local, dist=None, world=1):
    """eb_sample_blocks: 64 blocks (peak growth 0.1-0.8, so they stop after different step
    counts) on 8 slots; a freed slot takes the next block while the others keep denoising.
    The stand-in denoiser regenerates the occupied slots' logits on the device every iteration."""
    import ctypes

    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth
    import eb_synth.device as synth_dev

    stream = torch.cuda.current_stream(device)
    n, slots = 64, 8
    cfg = eb_synth.cfg3(B=n)
    recipe = synth_dev.Recipe.of(cfg)
    buf = torch.empty((slots, cfg.L, cfg.V), dtype=torch.int16, device=device)
    ws_bytes = eb.eb_blocks_workspace_bytes(slots, cfg.L, cfg.V, eb.EB_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    toks = torch.empty((n, cfg.L), dtype=torch.int32, device=device)
    steps = torch.empty(n, dtype=torch.int32, device=device)
    status = torch.empty(n, dtype=torch.int32, device=device)
    params = eb.eb_default_params(seed=0)

    def drive():
        return eb.eb_sample_blocks(params, slots, cfg.L, cfg.V, eb.EB_BF16, synth_dev.block_callback_address(),
                                   ctypes.addressof(recipe), buf, n, toks, steps, status, ws, ws_bytes,
                                   poll_every=8)

    drive()
    torch.cuda.synchronize()
    barrier(dist, local)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        start.record(stream)
        iters = drive()
        end.record(stream)
        torch.cuda.synchronize()
    barrier(dist, local)
    elapsed = start.elapsed_time(end) / 1e3
    value, slowest = aggregate(n, elapsed, world, dist, local)
    st = steps.cpu().numpy()
    return {
        "metric": BLOCKS_METRIC, "value": value, "unit": "blocks/s", "steps": n,
        "warmup": 1, "ms_per_step": slowest * 1e3 / n, "higher_is_better": True, "dtype": "f32",
        "config": {"workload": "block driver: 64 blocks x 256 positions x 262144 bf16, sigma 3, peak "
                               "U(0,4) + r s, r in (0.1, 0.2, 0.4, 0.8), up to 48 steps each, 8 slots",
                   "slots": slots, "iterations": iters},
        "canvas_steps_per_s": float(st.sum()) / slowest,
        "slot_occupancy": float(st.sum()) / (iters * slots),
        "steps_to_stop_mean": float(st.mean()),
        "stop_reasons": {str(k): int(v) for k, v in zip(*np.unique(status.cpu().numpy(), return_counts=True))},
        "gpu_launches": None,
        "clocks": clocks.summary(),
    }


# ------------------------------------------------------------------ adaptive loop workloads

LOOP_METRIC = ("EB adaptive denoising loop: canvas-steps/s over {B} canvas{es} x 256 x 262144 bf16 ({what}), "
               "stand-in denoiser included")


def measure_loop(cfg, label, runs, warm, device, local, dist=None, world=1):
    """The whole <= 48-step loop (eb_sample_canvas) over cfg.B canvases whose logits the seeded
    stand-in denoiser regenerates on the device every step; reports steps to stop per canvas and
    positions committed per step.  One 'step' of the metric is one canvas-step."""
    import ctypes

    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth.device as synth_dev

    stream = torch.cuda.current_stream(device)
    recipe = synth_dev.Recipe.of(cfg)
    buf = torch.empty((cfg.B, cfg.L, cfg.V), dtype=torch.int16, device=device)
    params = eb.eb_default_params(seed=int(cfg.seeds[0]))

    def loop(c):
        return c.run(params, synth_dev.callback_address(), ctypes.addressof(recipe), buf, poll_every=4)

    for _ in range(warm):
        loop(eb.Canvas(cfg.B, cfg.L, cfg.V, eb.EB_BF16, device=device))
    # fresh canvases made before the timed region; every loop is timed by its own events
    canv = [eb.Canvas(cfg.B, cfg.L, cfg.V, eb.EB_BF16, device=device) for _ in range(runs)]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(runs)]
    torch.cuda.synchronize()
    barrier(dist, local)
    with ClockSampler(local) as clocks:
        for c, (b, e) in zip(canv, ev):
            b.record(stream)
            loop(c)
            e.record(stream)
        torch.cuda.synchronize()
    barrier(dist, local)
    loop_ms = [b.elapsed_time(e) for b, e in ev]
    canvas_steps = sum(int(c.steps_taken.sum().item()) for c in canv)
    elapsed = sum(loop_ms) / 1e3
    c = canv[-1]
    value, slowest = aggregate(canvas_steps, elapsed, world, dist, local)
    st = c.steps_taken.cpu().numpy().tolist()
    com = c.committed_per_step.cpu().numpy()
    per_step = [[int(v) for v in row[:n]] for row, n in zip(com, st)]
    return {
        "metric": LOOP_METRIC.format(B=cfg.B, es="es" if cfg.B > 1 else "", what=label), "value": value,
        "unit": "canvas-steps/s", "steps": canvas_steps, "warmup": warm,
        "ms_per_step": slowest * 1e3 / canvas_steps, "higher_is_better": True, "dtype": "f32",
        "config": {"workload": f"adaptive loop ({label}): {cfg.B} canvas{'es' if cfg.B > 1 else ''} x 256 "
                               f"positions x 262144 bf16, sigma {cfg.sigma:g}, peak U({cfg.base_lo:g},"
                               f"{cfg.base_lo + cfg.base_scale:g}) + r s, r in {sorted(set(cfg.growth))}, "
                               "up to 48 steps, logits regenerated on the device every step",
                   "loops": runs},
        "loop_ms_median": float(np.median(loop_ms)),
        "steps_to_stop": st,
        "stop_reason": c.status.cpu().numpy().tolist(),
        "committed_per_step": per_step if cfg.B == 1 else None,
        "tokens_committed_per_step_mean": float(com[com > 0].mean()) if (com > 0).any() else 0.0,
        "tokens_committed_per_step_by_canvas": [float(cfg.L) / n for n in st],
        "gpu_launches": None,
        "clocks": clocks.summary(),
    }


# ------------------------------------------------------------------ all workloads in one run

def extras(args, device, local):
    """The per-workload records of the headline line, each measured here on the same GPU."""
    import dataclasses

    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth
    out = {}
    out["fused"] = measure_fused(4, 20, 3, 10, device, local)
    torch.cuda.empty_cache()
    out["fused1"] = measure_fused(1, 40, 3, 10, device, local)
    torch.cuda.empty_cache()
    out["loop_b1"] = measure_loop(eb_synth.cfg2(), "full adaptive loop, one canvas, peak growth 0.3", 5, 1,
                                  device, local)
    out["loop_b8"] = measure_loop(eb_synth.cfg3(), "mixed batch of eight, peak growth 0.1-0.8", 3, 1,
                                  device, local)
    out["loop_stop"] = measure_loop(eb_synth.cfg_stop(), "early stop, one canvas, sigma 1, peak growth 0.5", 5,
                                    1, device, local)
    torch.cuda.empty_cache()
    fp8 = argparse.Namespace(**{**vars(args), "logits": "fp8", "steps": 200, "warmup": 5})
    lk = logits_kind(fp8, eb, torch)
    m = run_single(fp8, lk, device, local, None, 1)
    peak, _ = measured_peaks()
    out["e4m3"] = {
        "metric": lk["metric"], "value": m["value"], "unit": "steps/s", "steps": m["K"],
        "ms_per_step": m["slowest"] * 1e3 / m["K"], "higher_is_better": True, "dtype": "f32",
        "config": {"workload": lk["workload"], "logits_dtype": "e4m3"},
        "roofline": {"bound": "hbm", "kernel": "k1_rowstats<e4m3>",
                     "achieved": lk["bytes"] / (m["k1"]["median_ms"] / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": lk["bytes"] / (m["k1"]["median_ms"] / 1e3) / 1e9 / peak,
                     "k1_ms_median": m["k1"]["median_ms"], "k1_ms_p10": m["k1"]["p10_ms"],
                     "k1_ms_p90": m["k1"]["p90_ms"], "k1_samples": m["k1"]["n"],
                     "bytes_per_launch": lk["bytes"]},
        "clocks": m["clocks"],
    }
    del m
    torch.cuda.empty_cache()
    out["blocks"] = measure_blocks(device, local)
    return out


def run_workload(args, rank, world, local):
    """`--workload NAME`: one of the other workloads as the printed line."""
    import torch

    import canvas_sampler_step_b300 as eb
    import eb_synth
    import eb_synth.device as synth_dev

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    eb.lib()
    synth_dev.lib()
    if args.workload in ("fused", "fused1"):
        FB = 1 if args.workload == "fused1" else 4
        out = measure_fused(FB, args.steps, args.warmup, args.e2e_steps, device, local, dist, world)
    elif args.workload in ("loop", "loop1", "stop"):
        cfg = {"loop": eb_synth.cfg3, "loop1": eb_synth.cfg2, "stop": eb_synth.cfg_stop}[args.workload]()
        label = {"loop": "mixed batch of eight, peak growth 0.1-0.8",
                 "loop1": "full adaptive loop, one canvas, peak growth 0.3",
                 "stop": "early stop, one canvas, sigma 1, peak growth 0.5"}[args.workload]
        out = measure_loop(cfg, label, max(1, args.steps // 200), max(1, args.warmup // 100), device, local,
                           dist, world)
    else:
        out = measure_blocks(device, local, dist, world)
    line = {"metric": out.pop("metric"), "value": out.pop("value"), "unit": out.pop("unit"), "n_gpus": world}
    line.update(out)
    line.update({"scaling": "weak", "vs_baseline": None,
                 "data": "synthetic (seeded Philox / Box-Muller inputs, eb_synth)"})
    line["config"]["parallelism"] = f"replicas x{world}"
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world, local)
    elif args.workload == "single":
        run_ours(args, rank, world, local)
    else:
        run_workload(args, rank, world, local)


if __name__ == "__main__":
    main()
