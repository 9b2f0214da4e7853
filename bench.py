"""Benchmark: one paged-KV decode step on GB300.

A step is one pass of the whole hot path over one batch: the append of this
step's token for every sequence (slot scatter), then paged decode attention
(block-table gather, TMA staging of K/V blocks, fused QK / online softmax / PV,
split-KV partials and the cross-split reduce).  By default the append is fused
into the decode kernel (decode_step); --two-call runs kv_cache_append and
paged_attn_decode as separate calls.  The timed region holds K steps back to
back between two CUDA events (inputs larger than L2); a batch whose KV fits in
twice the L2 size gets an L2 flush before every step and is timed step by
step.  The end-to-end leg adds every step's host copies through the same
public API.  The default workload is the
Llama-7B-shaped MHA decode batch (64 sequences, 32 q/kv heads, head_dim 128,
block_size 16, fp16, context lengths uniform in [512, 4096], blocks shuffled
over a 16384-block pool), with seeded synthetic inputs.

Prints ONE JSON line (rank 0).  `value` is decode-attention KV-read GB/s of the
whole job: algorithmic K+V bytes (sum_i L_i * Hkv * D * 2 * 2 per step, all
ranks) / max-over-ranks time of the timed steps.  The line's `workloads` object
holds the same step measured on the other workloads (tiny MHA, Llama-3-8B GQA,
long-context GQA, continuous batching with its two-call append time).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
    (N > 1: launch under torch.distributed.run; every rank runs an
     independent replica of the batch, no collective on the data path)
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
from dataclasses import replace

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from paged_kv_cache_268_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode-attention KV-read GB/s and % of GB300 HBM peak; seq-tokens/s"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "llama7b_mha"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, nominal
# the other workloads measured in the same run (``workloads`` in the JSON line)
OTHER_WORKLOADS = ("tiny_mha", "llama3_8b_gqa", "long_ctx_gqa", "cont_batch")
DTYPE_NAME = {W.F16: "f16", W.BF16: "bf16"}


# ---------------------------------------------------------------- helpers
def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["pkv", "reference"], default="pkv")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    p.add_argument("--kernel", type=int, default=0,
                   help="inner loop: 0 library's choice, 1 CUDA cores, 2 mma.sync, 3 tcgen05")
    p.add_argument("--num-seqs", type=int, default=0,
                   help="shrink the batch (and pool) for profiler captures; 0 = full workload")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--split-tokens", type=int, default=0)
    p.add_argument("--two-call", action="store_true",
                   help="time kv_cache_append + paged_attn_decode as two calls instead of "
                        "the fused decode_step")
    p.add_argument("--copy-bench", action="store_true",
                   help="also time pkv_copy_blocks (device->device, device->pinned host, "
                        "pinned host->device) on blocks of this workload's shape")
    p.add_argument("--graph", action="store_true",
                   help="capture one step in a CUDA graph and replay it (cuts host launch "
                        "overhead for small batches)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the per-workload measurements of the other four workloads")
    p.add_argument("--workload-seconds", type=float, default=0.25,
                   help="least device time of each other workload's timed region")
    return p.parse_args(argv)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def host_cpu() -> dict:
    """The host the CPU baseline runs on: logical CPUs and the CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith("model name"):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or None,
            "machine": platform.machine()}


def kernel_source_hash() -> str:
    csrc = os.path.join(ROOT, "paged_kv_cache_268_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, or None when missing or taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    entry = j.get(workload)
    if not entry or entry.get("kernel_source_sha") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_full_launch")


class ClockSampler:
    """nvidia-smi clocks/throttle sampler (started before, stopped after the
    timed region); keeps host timestamps so samples can be cut to the region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if not self.proc:
            return None
        inside = [p for t, p in self.samples if t0 <= t <= t1]
        window = "timed"
        if len(inside) < 3:
            inside = [p for t, p in self.samples if t <= t1]
            window = "warmup+timed"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for p in inside for k in range(4) if p[5 + k].lower() == "active"})
        power = [num(p[3]) for p in inside if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside), "window": window,
                "power_w_max": max(power) if power else None}


def job_totals(dist, device, elapsed_ms: float, units: dict):
    """Whole-job view of one timed region across replicas: the slowest rank's
    time (MAX) and the sum over ranks of each unit count (every rank runs its
    own seeded batch, so counts differ).  Without `dist` the local values."""
    if dist is None:
        return float(elapsed_ms), {k: float(v) for k, v in units.items()}
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    keys = sorted(units)
    u = torch.tensor([float(units[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), {k: float(v) for k, v in zip(keys, u.tolist())}


# ---------------------------------------------------------------- workload
def build_workload(args, rank: int, device):
    spec = W.WORKLOADS[args.workload]
    if args.num_seqs and args.num_seqs != spec.num_seqs:
        # same length distribution, heads and pool density; fewer sequences
        n = args.num_seqs
        largs = (tuple(spec.len_args[i % len(spec.len_args)] for i in range(n))
                 if spec.lens == "fixed" else spec.len_args)
        spec = replace(spec, name=f"{spec.name}/{n}", num_seqs=n, len_args=largs,
                       num_blocks=max(64, -(-spec.num_blocks * n // spec.num_seqs)))
    return W.make(spec, seed=args.seed + rank, device=device)


class OracleSampler:
    """Times the CPU oracle on bounded samples of (sequence, query head) rows
    of one workload.  The referenced K/V blocks are gathered to the host once;
    each run() then computes a random sample of rows sized to a time budget."""

    def __init__(self, w: W.Workload):
        import oracle  # test infrastructure: only the CPU-baseline / reference legs use it
        self.oracle = oracle
        self.w = w
        spec = w.spec
        nblk = -(-w.context_lens // spec.block_size)
        ids = np.concatenate([w.block_tables[i, :n] for i, n in enumerate(nblk)])
        uniq, inv = np.unique(ids, return_inverse=True)
        idx = torch.from_numpy(uniq.astype(np.int64)).to(w.k_cache.device)
        self.kc = W.bits(w.k_cache.index_select(0, idx))
        self.vc = W.bits(w.v_cache.index_select(0, idx))
        self.tables = np.full_like(w.block_tables, -1)
        k = 0
        for i, n in enumerate(nblk):
            self.tables[i, :n] = inv[k:k + n]
            k += n
        self.q = W.bits(w.q)
        mid = int(np.argsort(w.context_lens)[len(w.context_lens) // 2])
        t0 = time.perf_counter()
        self._rows(np.array([[mid, 0]], dtype=np.int32))
        self.per_row = max(time.perf_counter() - t0, 1e-5)

    def _rows(self, rows):
        w = self.w
        return self.oracle.decode_rows(rows, self.q, self.kc, self.vc, self.tables,
                                       w.context_lens, w.scale, w.spec.dtype)

    def run(self, target_s: float, seed: int = 0):
        """Returns (GB/s of KV rows read, description, seconds)."""
        spec = self.w.spec
        total = spec.num_seqs * spec.num_q_heads
        nrows = int(max(1, min(total, target_s / self.per_row)))
        flat = np.random.default_rng(seed).choice(total, size=nrows, replace=False)
        rows = np.stack([flat // spec.num_q_heads, flat % spec.num_q_heads], axis=1).astype(np.int32)
        t0 = time.perf_counter()
        self._rows(rows)
        dt = time.perf_counter() - t0
        # KV bytes a row reads: its L tokens of K and V for one kv head, shared by G q heads
        kv = float(self.w.context_lens[rows[:, 0]].astype(np.int64).sum()) * spec.head_dim * 4 / spec.group
        desc = (f"{nrows} of {total} (sequence, q head) rows of {spec.name}, "
                f"single-threaded fp64 C oracle, {dt:.2f} s")
        return kv / dt / 1e9, desc, dt


def copy_bench(pkv, spec, dev, stream, n_pairs=1024, reps=20):
    """GB/s of pkv_copy_blocks moving n_pairs whole blocks (K and V, every kv
    head): within the GPU pool, GPU -> pinned host pool, pinned host -> GPU."""
    shape = (4 * n_pairs, spec.num_kv_heads, spec.block_size, spec.head_dim)
    dt = torch.float16 if spec.dtype == W.F16 else torch.bfloat16
    gk, gv = torch.zeros(shape, dtype=dt, device=dev), torch.zeros(shape, dtype=dt, device=dev)
    hshape = (n_pairs,) + shape[1:]
    hk, hv = torch.zeros(hshape, dtype=dt).pin_memory(), torch.zeros(hshape, dtype=dt).pin_memory()
    rng = np.random.default_rng(0)
    src = rng.permutation(shape[0])[:n_pairs]
    dst = rng.permutation(np.setdiff1d(np.arange(shape[0]), src))[:n_pairs]
    ppairs = {"device_to_device": np.stack([src, dst], 1),
              "device_to_host": np.stack([src, rng.permutation(n_pairs)], 1),
              "host_to_device": np.stack([rng.permutation(n_pairs), dst], 1)}
    pools = {"device_to_device": (gk, gv, gk, gv), "device_to_host": (gk, gv, hk, hv),
             "host_to_device": (hk, hv, gk, gv)}
    nbytes = n_pairs * 2 * gk[0].numel() * gk.element_size()
    res = {"pairs": n_pairs, "bytes_per_call": nbytes}
    for name, pr in ppairs.items():
        p = torch.from_numpy(pr.astype(np.int32)).to(dev)
        for _ in range(3):
            pkv.copy_blocks(*pools[name], p, stream=stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            pkv.copy_blocks(*pools[name], p, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        res[name + "_gbs"] = nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    assert pkv.get_device_error() == 0
    # the copy engines on one contiguous run of the same size, for scale
    # (pinned host <-> device, cudaMemcpyAsync through torch)
    flat_d = torch.empty(nbytes // 2, dtype=dt, device=dev)
    flat_h = torch.empty(nbytes // 2, dtype=dt).pin_memory()
    for name, (a, b) in (("device_to_host", (flat_h, flat_d)), ("host_to_device", (flat_d, flat_h))):
        for _ in range(3):
            a.copy_(b, non_blocking=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(reps):
            a.copy_(b, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        res["memcpy_contiguous_" + name + "_gbs"] = nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9
    return res


def measure_workload(pkv, name: str, args, dev, stream, peak: float, l2_bytes: int,
                     sampler=None) -> dict:
    """One of the other workloads, measured the way the headline one is: the
    fused step (this step's token appended for every sequence inside the
    paged decode launch, then the split reduce), W warm-up steps, then at
    least K steps and at least --workload-seconds of device time back to back
    between two CUDA events (a batch whose KV fits in twice the L2 size gets
    an L2 flush before every step and is timed step by step).  The
    continuous-batching workload is also timed as two calls
    (kv_cache_append, then paged_attn_decode), with the append alone timed
    by events around it."""
    import math
    w = W.make(W.WORKLOADS[name], seed=args.seed, device=dev)
    spec = w.spec
    q, kc, vc = w.q, w.k_cache, w.v_cache
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    slots = torch.from_numpy(w.slot_mapping).to(dev)
    k_new, v_new = w.k_new, w.v_new
    out = torch.empty_like(q)
    maxL = w.max_context_len
    shape = pkv.decode_shape(q, kc, bt, maxL, 0, 0)
    plan = pkv.decode_plan(shape)
    ws = pkv.alloc_workspace(shape, dev)

    def fused():
        pkv.decode_step(q, k_new, v_new, kc, vc, bt, cl, w.scale, out, max_context_len=maxL,
                        workspace=ws, stream=stream)

    def append():
        pkv.kv_cache_append(k_new, v_new, slots, kc, vc, stream=stream)

    def decode():
        pkv.paged_attn_decode(q, kc, vc, bt, cl, w.scale, out, max_context_len=maxL,
                              workspace=ws, stream=stream)

    def two_call():
        append()
        decode()

    kv_bytes = w.kv_bytes()
    flush = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
             if kv_bytes < 2 * l2_bytes else None)

    def region(fn, n):
        """Device ms of n steps of fn (see the docstring for the L2 rule)."""
        if flush is None:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(n):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in ev)

    for _ in range(max(args.warmup, 3)):
        fused()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0
    est = max(region(fused, 5) / 5, 1e-3)
    n = int(min(20000, max(args.steps, math.ceil(args.workload_seconds * 1e3 / est))))
    if flush is not None:
        n = min(n, 2000)
    n0 = pkv.launch_count()
    t0 = time.time()
    ms = region(fused, n)
    t1 = time.time()
    launches = pkv.launch_count() - n0
    step_s = ms / n * 1e-3
    gbs = kv_bytes / step_s / 1e9
    entry = {
        "ms_per_step": ms / n, "steps": n, "kv_gbs": gbs, "frac": gbs / peak,
        "frac_of_nominal_hbm": gbs / NOMINAL_HBM_GBS,
        "seq_tokens_per_s": spec.num_seqs / step_s,
        "context_tokens_per_s": float(w.context_lens.sum()) / step_s,
        "kv_bytes_per_step": kv_bytes, "sum_context_len": int(w.context_lens.sum()),
        "config": {"num_seqs": spec.num_seqs, "q_heads": spec.num_q_heads,
                   "kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
                   "block_size": spec.block_size, "element_type": DTYPE_NAME[spec.dtype],
                   "pool_blocks": spec.num_blocks,
                   "context_lens": f"{spec.lens}{tuple(spec.len_args)[:4]}"},
        "plan": {"grid_ctas": plan.grid_ctas, "split_tokens": plan.split_tokens,
                 "num_splits": plan.num_splits,
                 "kernel_variant": ["cuda-core", "mma.sync", "tcgen05"][plan.variant]},
        "step": "decode_step: append of 1 token/seq fused into paged decode",
        "gpu_launches": launches,
        "l2": ("no flush: inputs larger than L2" if flush is None else
               f"flushed: {2 * l2_bytes / 1e6:.0f} MB written before every timed step; "
               "steps timed one by one"),
        "clocks": sampler.summary(t0, t1) if sampler else None,
    }
    if spec.share_prefix:
        unique = w.unique_kv_bytes()
        entry["unique_kv_bytes_per_step"] = unique
        entry["unique_kv_gbs"] = unique / step_s / 1e9
        entry["unique_frac"] = unique / step_s / 1e9 / peak
        for _ in range(max(args.warmup, 3)):
            two_call()
        torch.cuda.synchronize()
        ms2 = region(two_call, n)
        # the append alone: events around each call, median over <= 200 steps
        nb = min(n, 200)
        marks = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(nb)]
        for m in marks:
            if flush is not None:
                flush.zero_()
            m[0].record(stream)
            append()
            m[1].record(stream)
            decode()
            m[2].record(stream)
        torch.cuda.synchronize()
        assert pkv.get_device_error() == 0
        entry["two_call"] = {
            "ms_per_step": ms2 / n,
            "kv_gbs": kv_bytes / (ms2 / n * 1e-3) / 1e9,
            "unique_kv_gbs": unique / (ms2 / n * 1e-3) / 1e9,
            "append_us_median": 1e3 * statistics.median(m[0].elapsed_time(m[1]) for m in marks),
            "decode_us_median": 1e3 * statistics.median(m[1].elapsed_time(m[2]) for m in marks),
            "step": "kv_cache_append(1 token/seq) then paged_attn_decode, back to back",
        }
    del w, q, kc, vc, ws, flush
    torch.cuda.empty_cache()
    return entry


# ---------------------------------------------------------------- reference arm
def run_reference(args):
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    spec = W.WORKLOADS[args.workload]
    w = W.make(spec, seed=args.seed, device="cuda" if torch.cuda.is_available() else "cpu")
    sampler = OracleSampler(w)
    nsteps = args.steps + args.warmup
    per_step = min(args.cpu_seconds, 120.0 / max(nsteps, 1))   # whole run ~2 minutes at most
    rates, times, desc = [], [], ""
    for i in range(nsteps):
        gbs, desc, dt = sampler.run(per_step, seed=i)
        if i >= args.warmup:
            rates.append(gbs)
            times.append(dt)
    value = statistics.median(rates)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "num_seqs": spec.num_seqs,
                   "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
                   "head_dim": spec.head_dim, "block_size": spec.block_size,
                   "element_type": DTYPE_NAME[spec.dtype], "seed": args.seed},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": "per step: " + desc, **host_cpu()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- our arm
def run_pkv(args):
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from paged_kv_cache_268_gb300 import _binding as pkv
    from paged_kv_cache_268_gb300 import build as pkv_build
    if rank == 0 or not os.path.exists(pkv_build.LIB):
        pkv_build.build()
    if dist:
        dist.barrier()
    pkv.load_library()

    w = build_workload(args, rank, dev)
    spec = w.spec
    q = w.q
    kc, vc = w.k_cache, w.v_cache
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    slots = torch.from_numpy(w.slot_mapping).to(dev)
    k_new, v_new = w.k_new, w.v_new
    out = torch.empty_like(q)
    maxL = w.max_context_len
    shape = pkv.decode_shape(q, kc, bt, maxL, args.split_tokens, args.kernel)
    plan = pkv.decode_plan(shape)
    ws_buf = pkv.alloc_workspace(shape, dev)
    stream = torch.cuda.current_stream(dev)

    def step(k_in=k_new, v_in=v_new, s_in=slots, q_in=q, bt_in=bt, cl_in=cl, out_t=out):
        st = torch.cuda.current_stream(dev)     # the capture stream inside a CUDA graph
        if args.two_call:
            pkv.kv_cache_append(k_in, v_in, s_in, kc, vc, stream=st)
            pkv.paged_attn_decode(q_in, kc, vc, bt_in, cl_in, w.scale, out_t, max_context_len=maxL,
                                  split_tokens=args.split_tokens, kernel=args.kernel,
                                  workspace=ws_buf, stream=st)
        else:
            pkv.decode_step(q_in, k_in, v_in, kc, vc, bt_in, cl_in, w.scale, out_t,
                            max_context_len=maxL, split_tokens=args.split_tokens,
                            kernel=args.kernel, workspace=ws_buf, stream=st)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert pkv.get_device_error() == 0

    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.2 if sampler else 0)
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    graph = None
    per_replay = 0
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        c0 = pkv.launch_count()
        with torch.cuda.graph(graph):
            step()
        per_replay = pkv.launch_count() - c0     # kernels captured in one step
        graph.replay()
    torch.cuda.synchronize()

    def one_step(marks=None):
        """One timed step; `marks` = (before, between append and decode, after)
        events, recorded only in the breakdown pass."""
        if marks:
            marks[0].record(stream)
        if graph is not None:
            if marks:
                marks[1].record(stream)
            graph.replay()
        elif args.two_call:
            pkv.kv_cache_append(k_new, v_new, slots, kc, vc, stream=stream)
            if marks:
                marks[1].record(stream)
            pkv.paged_attn_decode(q, kc, vc, bt, cl, w.scale, out, max_context_len=maxL,
                                  split_tokens=args.split_tokens, kernel=args.kernel,
                                  workspace=ws_buf, stream=stream)
        else:
            if marks:
                marks[1].record(stream)
            step()
        if marks:
            marks[2].record(stream)

    # Inputs that fit in L2 would be timed hot: for them every timed step is
    # preceded by a write of twice the L2 size, and only the steps are timed.
    kv_bytes = w.kv_bytes()
    l2_bytes = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 132 * 2**20
    flush = (torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
             if kv_bytes < 2 * l2_bytes else None)

    def timed_loop(n):
        """n steps; returns the device time in ms.  Large inputs: back to back
        between two events (no events between steps, which would add their
        own gaps).  Inputs under 2x L2: an L2 flush before each step, outside
        the per-step events."""
        if flush is None:
            start.record(stream)
            for _ in range(n):
                one_step()
            end.record(stream)
            torch.cuda.synchronize()
            return start.elapsed_time(end)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            one_step()
            e1.record(stream)
        torch.cuda.synchronize()
        return sum(e0.elapsed_time(e1) for e0, e1 in ev)

    # The timed region.
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = pkv.launch_count()
    t_host0 = time.time()
    loop_ms = timed_loop(K)
    t_host1 = time.time()
    # launches made through the library (a graph replays its captured kernels
    # without calling the library)
    launches = pkv.launch_count() - n0 if graph is None else per_replay * K
    if dist:
        dist.barrier()
    total_ms = loop_ms
    assert pkv.get_device_error() == 0
    hot = None
    if flush is not None:
        # the same steps back to back with a warm L2, for reference
        start.record(stream)
        for _ in range(K):
            one_step()
        end.record(stream)
        torch.cuda.synchronize()
        hot_ms = start.elapsed_time(end) / K
        hot = {"ms_per_step": hot_ms, "value": kv_bytes / (hot_ms * 1e-3) / 1e9, "unit": UNIT}

    # Per-step breakdown (median / P90 and the append share), after the timed
    # region: each step bracketed by events.
    nb = min(K, 200)
    marks = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(nb)]
    for i in range(nb):
        if flush is not None:
            flush.zero_()
        one_step(marks[i])
    torch.cuda.synchronize()
    decode_ms = [m[1].elapsed_time(m[2]) for m in marks]
    append_ms = [m[0].elapsed_time(m[1]) for m in marks]

    # K+V bytes of the distinct cache rows a step touches (a shared prefix
    # block counted once): what HBM has to deliver when L2 serves the repeats
    unique_bytes = w.unique_kv_bytes()
    total_ms, job = job_totals(dist, dev, total_ms,
                               {"kv_bytes": kv_bytes, "seqs": spec.num_seqs,
                                "ctx_tokens": int(w.context_lens.sum()),
                                "unique_kv_bytes": unique_bytes})
    ms_per_step = total_ms / K
    value = job["kv_bytes"] * K / (total_ms * 1e-3) / 1e9
    peak, peak_src = measured_peak()
    # this rank's average step (decode kernel + split reduce, append fused)
    # over the timed region
    achieved = kv_bytes * K / (loop_ms * 1e-3) / 1e9

    # end-to-end through the public API with pinned host buffers: every step
    # copies its inputs host->device, runs append + decode and reads its output
    # back.  As a serving loop would, the copies run on a second stream and
    # overlap the neighbouring steps' kernels: step i+1's inputs go up and
    # step i's output comes down while the GPU computes (inputs and outputs
    # are double-buffered).  The timed region spans every copy of every step.
    e2e = None
    if not args.no_e2e:
        h_q = q.cpu().pin_memory()
        h_k, h_v = k_new.cpu().pin_memory(), v_new.cpu().pin_memory()
        h_slots = slots.cpu().pin_memory()
        h_bt, h_cl = bt.cpu().pin_memory(), cl.cpu().pin_memory()
        hosts = [h_q, h_k, h_v, h_slots, h_bt, h_cl]
        sets = [[torch.empty_like(t, device=dev) for t in (q, k_new, v_new, slots, bt, cl)]
                for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        h_outs = [torch.empty_like(h_q).pin_memory() for _ in range(2)]
        up = [0, 1, 2, 4, 5] + ([3] if args.two_call else [])  # the fused step derives the slots
        h2d = sum(hosts[j].numel() * hosts[j].element_size() for j in up)
        d2h = h_outs[0].numel() * h_outs[0].element_size()
        xs = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        Ke = max(10, min(K, 500))

        def run_e2e(n):
            in_ready, computed, drained = [ev(), None], [None, None], [None, None]
            with torch.cuda.stream(xs):
                xs.wait_stream(stream)
                for j in up:
                    sets[0][j].copy_(hosts[j], non_blocking=True)
                in_ready[0].record(xs)
            for i in range(n):
                b = i & 1
                stream.wait_event(in_ready[b])
                if drained[b] is not None:
                    stream.wait_event(drained[b])        # out[b] of step i-2 is on the host
                dq, dk, dv, dsl, dbt, dcl = sets[b]
                step(dk, dv, dsl, dq, dbt, dcl, outs[b])
                computed[b] = ev()
                computed[b].record(stream)
                with torch.cuda.stream(xs):
                    if i + 1 < n:
                        nb = b ^ 1
                        if i >= 1:
                            xs.wait_event(computed[nb])  # step i-1 is done with set nb
                        for j in up:
                            sets[nb][j].copy_(hosts[j], non_blocking=True)
                        in_ready[nb] = ev()
                        in_ready[nb].record(xs)
                    xs.wait_event(computed[b])
                    h_outs[b].copy_(outs[b], non_blocking=True)
                    drained[b] = ev()
                    drained[b].record(xs)
            stream.wait_stream(xs)

        run_e2e(4)
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        s0.record(stream)
        run_e2e(Ke)
        s1.record(stream)
        torch.cuda.synchronize()
        e_ms, ejob = job_totals(dist, dev, s0.elapsed_time(s1), {"kv_bytes": kv_bytes})
        ref_out = torch.empty_like(out)
        step(out_t=ref_out)
        torch.cuda.synchronize()
        assert torch.equal(h_outs[(Ke - 1) & 1].view(torch.int16), ref_out.cpu().view(torch.int16))
        e2e = {"value": ejob["kv_bytes"] * Ke / (e_ms * 1e-3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
               "ms_per_step": e_ms / Ke,
               "copies": "pinned host <-> device on a second stream, overlapping the "
                         "neighbouring steps' kernels (double-buffered inputs and outputs)"}
        if flush is not None:
            e2e["l2"] = "not flushed: the steps run back to back and the KV fits in L2"

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    copy_res = copy_bench(pkv, spec, dev, stream) if args.copy_bench else None
    cpu = None
    if not args.no_cpu_baseline:
        gbs, desc, _ = OracleSampler(w).run(args.cpu_seconds)
        cpu = {"value": gbs, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": desc,
               **host_cpu()}

    # The other four workloads, each measured on its own in this process.
    others = None
    if not args.no_workloads and not args.num_seqs:
        others = {name: measure_workload(pkv, name, args, dev, stream, peak, l2_bytes, sampler)
                  for name in OTHER_WORKLOADS if name != args.workload}
    if sampler:
        sampler.stop()
    clocks = sampler.summary(t_host0, t_host1) if sampler else None
    traffic = recorded_traffic(spec.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_NAME[spec.dtype],
        "data": "synthetic",
        "config": {"workload": spec.name, "num_seqs": spec.num_seqs,
                   "q_heads": spec.num_q_heads, "kv_heads": spec.num_kv_heads,
                   "head_dim": spec.head_dim, "block_size": spec.block_size,
                   "pool_blocks": spec.num_blocks, "context_lens": f"{spec.lens}{tuple(spec.len_args)}",
                   "sum_context_len": int(w.context_lens.sum()), "seed": args.seed,
                   "step": ("kv_cache_append(1 token/seq) + paged_attn_decode" if args.two_call
                            else "decode_step: append of 1 token/seq fused into paged decode"),
                   "schedule": "partitions",
                   "grid_ctas": plan.grid_ctas,
                   "split_tokens": plan.split_tokens, "num_splits": plan.num_splits,
                   "kernel_variant": ["cuda-core", "mma.sync", "tcgen05"][plan.variant],
                   "l2": (f"no flush: inputs larger than L2 ({kv_bytes / 1e9:.2f} GB of KV per step "
                          f"vs {l2_bytes / 1e6:.0f} MB L2)" if flush is None else
                          f"flushed: {2 * l2_bytes / 1e6:.0f} MB written before every timed step "
                          f"(KV per step {kv_bytes / 1e6:.2f} MB fits in L2); steps timed one by one"),
                   "parallelism": f"replicas x{ws}",
                   "cuda_graph": bool(args.graph)},
        "pct_hbm_peak": value / ws / peak,
        "frac_of_nominal_hbm": value / ws / NOMINAL_HBM_GBS,
        "nominal_hbm_gbs": NOMINAL_HBM_GBS,
        "seq_tokens_per_s": job["seqs"] * K / (total_ms * 1e-3),
        "context_tokens_per_s": job["ctx_tokens"] * K / (total_ms * 1e-3),
        "unique_kv_bytes_per_step": unique_bytes,
        "unique_kv_gbs": job["unique_kv_bytes"] * K / (total_ms * 1e-3) / 1e9,
        "decode_ms_median": statistics.median(decode_ms),
        "decode_ms_p90": float(np.percentile(decode_ms, 90)),
        "append_us_median": 1e3 * statistics.median(append_ms) if args.two_call else None,
        "hot_cache": hot,
        "roofline": {"bound": "hbm",
                     "kernel": ("paged_attn_decode" if args.two_call else "decode_step")
                               + " (decode kernel + split reduce)",
                     "achieved": achieved, "peak": peak, "peak_source": peak_src,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": kv_bytes},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "block_copy": copy_res,
        "clocks": clocks,
        "workloads": others,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_pkv(args)


if __name__ == "__main__":
    sys.exit(main())
