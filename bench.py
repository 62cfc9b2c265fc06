"""Benchmark of the TBE hot path on GB300: forward + backward (transpose, sort,
run-length encoding, segment reduction, fused optimizer update) per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config 4] [--extra 2,3,5] [--index-dtype int64] [--no-e2e]
                  [--no-cpu-baseline]

Prints one JSON line on rank 0.  The headline workload (default) is the
hot-row backward stress case: T=16 bf16 tables of 5M rows x 128, B=65536,
pooling factor 32, Zipf(1.2) indices, row-wise Adagrad.  The other workloads
named by --extra are measured in the same run with the same step counts and
reported under "workloads".  Timing: CUDA events on the launching stream
around each step, L2 flushed (256 MiB write) before every step outside the
timed interval, W untimed warm-up steps, barrier + synchronize around the K
timed steps; ms_per_step is the median of the K per-step intervals, max over
ranks.  Under torchrun every rank runs its own replica (the path does not
shard: weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
ELEM = {"f32": 4, "f16": 2, "bf16": 2}
METRIC = "TBE fwd / fwd+bwd+update lookups/sec and HBM GB/s (% of GB300 roofline), 1 GPU"
# the kernels each call consists of (the first is its main one)
DOMINANT_KERNELS = {
    "forward": "fwd_pool_kernel (+ fwd_long_kernel, hist_kernel)",
    "prepare": "keys_kernel, upsweep/scan/downsweep per radix pass, run-length and chunk kernels",
    "apply": "apply_class_kernel per backward class (+ dense_mma_kernel, dense_update_kernel)",
}

# the sources of each call's kernels (a traffic profile is valid while they
# are unchanged)
_CSRC = "recommender_sparse_embeddings_gb300/csrc/"
KERNEL_FILES = {
    "forward": [_CSRC + "forward.cu", _CSRC + "hist.cu", _CSRC + "tbe_internal.cuh"],
    "prepare": [_CSRC + "prepare.cu", _CSRC + "tbe_internal.cuh"],
    "apply": [_CSRC + "apply.cu", _CSRC + "dense.cu", _CSRC + "tbe_internal.cuh"],
}


def kernel_sources_sha256(segment: str) -> str:
    """sha256 over the call's kernel sources, in the listed order."""
    h = hashlib.sha256()
    for f in KERNEL_FILES[segment]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def reduce_max(value: float, device) -> float:
    """Max of a host float over all ranks (identity when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, device) -> float:
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def wants_length_order(specs, mode: str) -> bool:
    """TBE_FLAG_LENGTH_ORDER as a caller who knows the batch's length law
    would set it: on for uniform lengths over a wide range (where it was
    measured faster), off for fixed or Poisson lengths (where it was not)."""
    if mode != "auto":
        return mode == "on"
    for sp in specs:
        law = sp.length
        if law[0] == "uniform" and law[2] >= 4 * max(law[1], 1):
            return True
    return False


def barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


# ------------------------------------------------------------------ bytes

def algorithmic_bytes(specs, batch_lengths, N, B, T, idx_bytes, weights, optimizer, U, passes):
    """Algorithmic bytes per step, by segment (the formula stated with the
    workload: gathered rows, indices/offsets/weights, outputs; backward adds
    the gradient rows gathered per lookup, the sort traffic and the
    read-modify-write of unique rows and optimizer state)."""
    per_table_lookups = batch_lengths.view(T, B).sum(1).tolist()
    gathered = sum(n * s.dim * ELEM[s.dtype] for n, s in zip(per_table_lookups, specs))
    total_d = sum(s.dim for s in specs)
    out_bytes = B * total_d * 4
    fwd = gathered + N * idx_bytes + (T * B + 1) * idx_bytes + (N * 4 if weights else 0) + out_bytes
    # transpose + sort + run-length: index/offset reads, key/bag (+scale) writes,
    # each radix pass reads and writes (key, value), run-length reads keys and
    # writes (uniq, runstart)
    scale = 4 if weights else 0
    prep = (N * idx_bytes + (T * B + 1) * idx_bytes + N * (4 + 4 + scale)
            + passes * N * 16 - N * 4 + N * 4 + U * 8)
    grad_rows = sum(n * s.dim * 4 for n, s in zip(per_table_lookups, specs))
    avg_row = sum(s.dim * ELEM[s.dtype] for s in specs) / len(specs)
    apply = grad_rows + N * (4 + 4 + scale) + U * 8 + 2 * U * avg_row + (
        2 * U * 4 if optimizer == "adagrad" else 0)
    return dict(forward=fwd, prepare=prep, apply=apply, step=fwd + prep + apply)


def wgrad_bytes(specs, batch_lengths, N, B, T, idx_bytes):
    """Algorithmic bytes of the per-sample weight gradient: the looked-up rows,
    indices and offsets (as the forward pass), the upstream gradient read once
    and one fp32 result per lookup."""
    per_table_lookups = batch_lengths.view(T, B).sum(1).tolist()
    gathered = sum(n * s.dim * ELEM[s.dtype] for n, s in zip(per_table_lookups, specs))
    total_d = sum(s.dim for s in specs)
    return gathered + N * idx_bytes + (T * B + 1) * idx_bytes + B * total_d * 4 + N * 4


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every period_ms) read by a thread; summary() keeps
    the samples taken between mark_start() and mark_end()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.samples = []  # (host time, line)
        self.t0 = self.t1 = None

    def __enter__(self):
        import threading

        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self

        def reader():
            for line in self.proc.stdout:
                if line.strip():
                    self.samples.append((time.perf_counter(), line))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        deadline = time.perf_counter() + 5.0  # wait for the first sample
        while not self.samples and time.perf_counter() < deadline:
            time.sleep(0.02)
        return self

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)
        return False

    def summary(self, window=None):
        """Median SM clock, max clock and throttle reasons seen between
        mark_start() and mark_end() (or inside `window` = (t0, t1))."""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        w0, w1 = window if window is not None else (self.t0, self.t1)
        t0 = w0 if w0 is not None else -1e30
        t1 = (w1 + 0.1) if w1 is not None else 1e30
        for ts, l in self.samples:
            if not (t0 <= ts <= t1):
                continue
            parts = [p.strip() for p in l.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- profile

def profile_traffic(segment: str, cfg, T: int):
    """DRAM bytes of one call (all its kernels) on this workload, from the
    committed ncu summary profiles/launches_traffic_<workload>.md, or None if
    there is none (for this workload and table count) or a kernel source
    changed since."""
    path = os.path.join(ROOT, "profiles", f"launches_traffic_{cfg.name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    t = re.search(r"^tables:\s*([0-9]+)", text, re.M)
    m = re.search(r"^traffic\[" + re.escape(segment) + r"\]:\s*([0-9.eE+]+)\s+sha256=([0-9a-f]+)", text, re.M)
    if not m or not t or int(t.group(1)) != T:
        return None
    if kernel_sources_sha256(segment) != m.group(2):
        return None
    return float(m.group(1))


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback (6.8 TB/s)"


# ------------------------------------------------------------ CPU baseline

class OracleSample:
    """A bounded sample of the workload for the CPU oracle (as it stands): the
    first `tables_in_sample` tables with the full B and the same laws.  One
    step = oracle forward + oracle backward (with the workload's optimizer)."""

    def __init__(self, cfg, tables_in_sample: int = 2, bags: int = 0, threads: int = 1):
        import numpy as np

        total_tables = len(workloads.realize_tables(cfg))
        if bags and bags < cfg.B:
            cfg = cfg.scaled(B=bags)  # same rows and laws, fewer bags per table
        self.cfg = cfg
        specs = workloads.realize_tables(cfg)[:tables_in_sample]
        tabs_t = workloads.make_tables(cfg, "cpu", specs)
        batch = workloads.make_batch(cfg, "cpu", torch.int64, specs)
        self.names = [s.dtype for s in specs]
        self.tabs = [t.numpy() if t.dtype == torch.float32
                     else t.view(torch.int16).numpy().view(np.uint16) for t in tabs_t]
        self.ind, self.off = batch.indices.numpy(), batch.offsets.numpy()
        self.w = None if batch.weights is None else batch.weights.numpy()
        self.g = workloads.make_grad(cfg, "cpu", specs).numpy()
        self.state = (np.zeros(sum(s.rows for s in specs), np.float32)
                      if cfg.optimizer == "adagrad" else None)
        self.N = batch.N
        self.threads = threads
        self.sample = (f"{tables_in_sample} of {total_tables} tables, "
                       f"B={cfg.B}, {batch.N} lookups per fwd+bwd step")

    def step(self) -> float:
        import oracle

        # the pinned one-thread build, or the OpenMP timing build on `threads` cores
        if self.threads == 1:
            oracle.use_plain_build()
        else:
            oracle.use_timing_build(self.threads)
        c = self.cfg
        t0 = time.perf_counter()
        oracle.forward(self.tabs, self.names, self.ind, self.off, c.B, weights=self.w,
                       pooling=c.pooling)
        oracle.backward(self.tabs, self.names, self.ind, self.off, c.B, self.g, c.optimizer, c.lr,
                        eps=c.eps, weights=self.w, pooling=c.pooling, state=self.state)
        return time.perf_counter() - t0


def backward_classes(specs) -> int:
    """Backward apply launches one kernel per (dtype, row shape) class; the
    bench's tables and gradient are aligned, so the shape is the dim when it
    is 32, 64, 128 or 256, and element-wise otherwise."""
    return len({(s.dtype, s.dim if s.dim in (32, 64, 128, 256) else 0) for s in specs})


def _mean_bag_length(spec) -> float:
    kind = spec.length[0]
    if kind == "fixed":
        return float(spec.length[1])
    if kind == "poisson":
        return float(spec.length[1])
    return (spec.length[1] + spec.length[2]) / 2.0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_oracle_run(cfg, seconds: float = 10.0, threads: int = 1, sample=None):
    """The oracle as it stands on a bounded sample of the workload: one core
    (the pinned build) or `threads` cores (the OpenMP timing build of the
    same source).  Runs whole steps until `seconds` of CPU time pass."""
    s = sample if sample is not None else OracleSample(cfg)
    s.threads = threads
    s.step()  # first touch of the sample's memory, untimed
    steps, el = 0, 0.0
    while steps == 0 or el < seconds:
        el += s.step()
        steps += 1
    return {"lookups": s.N * steps, "seconds": el, "steps": steps,
            "sample": s.sample + f", {steps} steps on {threads} thread(s)", "oracle_sample": s}


# ---------------------------------------------------------------- our arm

def measure(tbe, cfg_id, args, dev, clk, headline):
    """One workload: generate, warm up, time K steps (forward + preparation,
    then apply), time each call alone, and (headline only) the end-to-end
    run through pinned host buffers.  Returns the workload's record."""
    world, rank, _ = dist_env()
    cfg = workloads.get_config(cfg_id)
    specs = workloads.realize_tables(cfg)
    if args.tables:
        specs = specs[:args.tables]
    idx_dtype = torch.int64 if args.index_dtype == "int64" else torch.int32
    tables = workloads.make_tables(cfg, dev, specs)
    batch = workloads.make_batch(cfg, dev, idx_dtype, specs)
    grad = workloads.make_grad(cfg, dev, specs)
    T, B, N = len(specs), cfg.B, batch.N
    length_order = wants_length_order(specs, args.length_order)
    # the small tables' forward: the histogram path where the workload
    # prescribes it (auto), else the library's default (the gather)
    histogram = cfg.histogram_forward if args.histogram == "auto" else args.histogram == "on"
    flags = (tbe.TBE_FLAG_NO_HISTOGRAM if args.no_histogram else 0) | (
        tbe.TBE_FLAG_SORTED_BACKWARD if args.sorted_backward else 0) | (
        tbe.TBE_FLAG_FORCE_HISTOGRAM if histogram else 0) | (
        tbe.TBE_FLAG_LENGTH_ORDER if length_order else 0)
    h = tbe.tbe_create(tables, cfg.pooling, flags)
    ws = tbe.make_workspace(h, N, B, dev)
    out = torch.empty((B, h.total_dim), dtype=torch.float32, device=dev)
    state = (torch.zeros(h.total_rows, dtype=torch.float32, device=dev)
             if cfg.optimizer == "adagrad" else None)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    ind, off, w = batch.indices, batch.offsets, batch.weights

    def fwd():
        tbe.tbe_forward(h, ind, off, B, w, out)

    def prep():
        tbe.tbe_backward_prepare(h, ind, off, B, ws, w)

    def fwd_prep():
        # forward and the backward preparation of the same batch, side by side
        tbe.tbe_forward_prepare(h, ind, off, B, ws, w, out)

    def apply(g=grad):
        tbe.tbe_backward_apply(h, N, B, g, ws, cfg.optimizer, cfg.lr, cfg.eps, state)

    for _ in range(args.warmup):
        flush.zero_()
        fwd_prep(); apply()
    torch.cuda.synchronize()
    rc = tbe.tbe_get_error(h)
    if rc != tbe.TBE_OK:
        raise RuntimeError(f"device error during warm-up: {tbe.tbe_strerror(rc)}")
    run_fp, run_ap = fwd_prep, apply
    if args.graph:
        # the same calls captured once as two CUDA graphs (the library's side
        # streams fork from and join back into the capturing stream)
        g_fp, g_ap = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_fp):
            fwd_prep()
        with torch.cuda.graph(g_ap):
            apply()
        torch.cuda.synchronize()
        run_fp, run_ap = g_fp.replay, g_ap.replay
        for _ in range(args.warmup):
            flush.zero_()
            run_fp(); run_ap()
        torch.cuda.synchronize()

    # timed region: one step = forward + preparation (concurrent), then apply
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize()
    t_start = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        e = ev[k]
        e[0].record(stream); run_fp()
        e[1].record(stream); run_ap()
        e[2].record(stream)
    torch.cuda.synchronize()
    t_end = time.perf_counter()
    barrier()
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    seg_lists = {"forward+prepare": [e[0].elapsed_time(e[1]) for e in ev],
                 "apply": [e[1].elapsed_time(e[2]) for e in ev]}
    med_ms = reduce_max(statistics.median(step_ms), dev)
    mean_ms = reduce_max(sum(step_ms) / len(step_ms), dev)
    units = reduce_sum(float(N), dev)  # lookups of one step over all ranks
    rc = tbe.tbe_get_error(h)
    if rc != tbe.TBE_OK:
        raise RuntimeError(f"device error in timed region: {tbe.tbe_strerror(rc)}")

    # per-call breakdown (a separate run, each call timed alone; medians)
    nb_steps = min(args.steps, 200)
    evb = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nb_steps)]
    for k in range(nb_steps):
        flush.zero_()
        e = evb[k]
        e[0].record(stream); fwd()
        e[1].record(stream); prep()
        e[2].record(stream); apply()
        e[3].record(stream)
    torch.cuda.synchronize()
    brk = {name: statistics.median(e[i].elapsed_time(e[i + 1]) for e in evb)
           for i, name in enumerate(("forward", "prepare", "apply"))}

    # per-sample weight gradient (weighted batches): timed alone, after a flush
    wg_ms = None
    if w is not None:
        gw_out = torch.empty(N, dtype=torch.float32, device=dev)
        evw = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(nb_steps)]
        for k in range(nb_steps):
            flush.zero_()
            evw[k][0].record(stream)
            tbe.tbe_per_sample_weight_grad(h, ind, off, B, grad, gw_out)
            evw[k][1].record(stream)
        torch.cuda.synchronize()
        wg_ms = statistics.median(a.elapsed_time(b) for a, b in evw)
        rc = tbe.tbe_get_error(h)
        if rc != tbe.TBE_OK:
            raise RuntimeError(f"device error in the weight gradient: {tbe.tbe_strerror(rc)}")

    # U (distinct keys) for the byte count: read once after the run; the
    # dense-backward tables' lookups are not sorted, so their distinct rows
    # are counted here
    lay = tbe.tbe_backward_workspace_layout(h, N, B)
    U = int(ws[lay.num_unique:lay.num_unique + 4].view(torch.int32).item())
    offs = off.to(torch.int64).cpu()
    paths = tbe.tbe_table_paths(h)
    bpaths = tbe.tbe_backward_paths(h)
    for t, p in enumerate(bpaths):
        if p == "dense":
            lo, hi = int(offs[t * B]), int(offs[(t + 1) * B])
            U += int(torch.unique(ind[lo:hi]).numel())
    # compulsory bytes (each distinct row, the gradient and the batch once):
    # the floor under the formula's bytes, which count every gathered row
    u_row_bytes = 0
    for t, sp in enumerate(specs):
        lo, hi = int(offs[t * B]), int(offs[(t + 1) * B])
        u_t = int(torch.unique(ind[lo:hi]).numel()) if hi > lo else 0
        u_row_bytes += u_t * sp.dim * ELEM[sp.dtype]
    total_d = sum(sp.dim for sp in specs)
    ib = idx_dtype.itemsize
    scale_b = 4 if (w is not None or cfg.pooling == "mean") else 0
    compulsory = {
        "forward": u_row_bytes + N * ib + (T * B + 1) * ib + (N * 4 if w is not None else 0) + B * total_d * 4,
        "apply": B * total_d * 4 + N * (4 + 4 + scale_b) + U * 8 + 2 * u_row_bytes
                 + (2 * U * 4 if cfg.optimizer == "adagrad" else 0),
    }
    # radix passes of the sort: 8-bit digits, or 9-bit ones when they save a pass
    key_bits = max(1, h.total_rows.bit_length())
    passes = min((key_bits + 7) // 8, (key_bits + 8) // 9)
    nbytes = algorithmic_bytes(specs, batch.lengths, N, B, T, idx_dtype.itemsize, w is not None,
                               cfg.optimizer, U, passes)
    nbytes["forward+prepare"] = nbytes["forward"] + nbytes["prepare"]
    value = units / (med_ms / 1e3)
    peak, peak_src = measured_hbm_peak()
    seg_ms = {k: statistics.median(v) for k, v in seg_lists.items()}
    # roofline of the dominant call (forward, prepare or apply: the one that
    # takes longest alone).  The apply is timed inside the timed region on the
    # caller's stream (its side streams join back before the closing event);
    # forward and prepare overlap there, so theirs come from the per-call run.
    call_ms = dict(brk)
    call_ms["apply"] = seg_ms["apply"]
    dominant = max(call_ms, key=call_ms.get)
    achieved = nbytes[dominant] / (call_ms[dominant] / 1e3) / 1e9
    timing_src = ("timed region, CUDA events on the caller's stream, median of the steps" if dominant == "apply"
                  else "per-call run, CUDA events on the caller's stream, median of the steps")
    traffic = profile_traffic(dominant, cfg, T)
    # our kernels per step: forward (gather pool if any gather table, long
    # bags, one histogram launch per dtype with histogram tables); prepare
    # (bag marks, [compaction], keys, per radix pass [upsweep] + scan +
    # downsweep, run-length count/scan/write, chunk count/scan/write); apply
    # (one per backward class of the sorted-path tables, dense sums + update)
    hist_dtypes = {s.dtype for s, p in zip(specs, paths) if p == "histogram"}
    dense = "dense" in bpaths  # small tables' dense backward
    fwd_launches = (1 if any(p != "histogram" for p in paths) else 0) + 1 + len(hist_dtypes)
    prep_launches = 2 + (1 if dense else 0) + 2 * passes + (passes if dense else passes - 1) + 6
    sorted_specs = [s for s, p in zip(specs, bpaths) if p == "sorted"]
    apply_launches = backward_classes(sorted_specs) + (2 if dense else 0)
    launches_per_step = fwd_launches + prep_launches + apply_launches

    rec = {
        "value": value,
        "unit": "lookups/s",
        "ms_per_step": med_ms,
        "ms_per_step_mean": mean_ms,
        "timed_region_s": t_end - t_start,
        "dtype": "f32" if all(sp.dtype == "f32" for sp in specs) else "mixed(f32 accumulate)",
        "paths": sorted(set(paths)),
        "backward_paths": sorted(set(bpaths)),
        "config": {"workload": cfg.description + (f" (first {T} of the tables)" if args.tables else ""),
                   "config_id": cfg.cfg_id, "T": T, "B": B, "N_lookups": N, "unique_rows": U,
                   "index_dtype": args.index_dtype, "optimizer": cfg.optimizer,
                   "parallelism": f"replicas x{world}",
                   "launch": "CUDA graph replay" if args.graph else "stream launches",
                   "bag_order": "by length (TBE_FLAG_LENGTH_ORDER)" if length_order else "index order",
                   "small_table_forward": "tensor-core histogram" if histogram else "gather",
                   "l2": "flushed (256 MiB write) before every step, outside the timed interval"},
        "fwd": {"lookups_per_s": N / (brk["forward"] / 1e3),
                "gbs": nbytes["forward"] / (brk["forward"] / 1e3) / 1e9,
                "frac": nbytes["forward"] / (brk["forward"] / 1e3) / 1e9 / peak,
                "ms": brk["forward"]},
        "wgrad": None if wg_ms is None else {
            "ms": wg_ms, "bytes": wgrad_bytes(specs, batch.lengths, N, B, T, idx_dtype.itemsize),
            "gbs": wgrad_bytes(specs, batch.lengths, N, B, T, idx_dtype.itemsize) / (wg_ms / 1e3) / 1e9,
            "frac": wgrad_bytes(specs, batch.lengths, N, B, T, idx_dtype.itemsize) / (wg_ms / 1e3) / 1e9 / peak,
            "note": "per-sample weight gradient, timed alone outside the step"},
        "step_gbs": nbytes["step"] / (med_ms / 1e3) / 1e9,
        "segments_ms": seg_ms,
        "breakdown_ms_sequential": brk,
        "algorithmic_bytes": nbytes,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "dram_frac": None if traffic is None else traffic / (call_ms[dominant] / 1e3) / 1e9 / peak,
                     "kernel": DOMINANT_KERNELS[dominant], "call": dominant,
                     "ms_per_launch": call_ms[dominant], "bytes_per_launch": nbytes[dominant],
                     "timing": timing_src, "peak_source": peak_src,
                     "segment_fracs": {k: nbytes[k] / (v / 1e3) / 1e9 / peak for k, v in seg_ms.items()},
                     "compulsory": {k: {"bytes": compulsory[k],
                                        "frac": compulsory[k] / (call_ms[k] / 1e3) / 1e9 / peak}
                                    for k in ("forward", "apply")}},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary((t_start, t_end)),
    }

    # end-to-end through the public API: inputs from pinned host memory every
    # step, pooled output read back every step.  Two sets of device buffers:
    # the next step's inputs copy in while this step computes, and this
    # step's output copies out while the next one starts.
    rec["e2e"] = None
    if headline and not args.no_e2e:
        h_ind = ind.cpu().pin_memory()
        h_off = off.cpu().pin_memory()
        h_w = None if w is None else w.cpu().pin_memory()
        h_grad = grad.cpu().pin_memory()
        h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        bufs = [dict(ind=torch.empty_like(ind), off=torch.empty_like(off),
                     w=None if w is None else torch.empty_like(w), grad=torch.empty_like(grad),
                     out=torch.empty_like(out)) for _ in range(2)]
        # copies in on two streams (the batch on one, the upstream gradient on
        # the other, so two copy engines work at once), out on a third
        copy_in, copy_in2, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # buffer i holds its step's inputs
        ev_used = [torch.cuda.Event() for _ in range(2)]   # buffer i's step has read its inputs
        ev_out = [torch.cuda.Event() for _ in range(2)]    # buffer i's output is on the host

        def copy_inputs(i):
            copy_in.wait_event(ev_used[i])
            copy_in2.wait_event(ev_used[i])
            with torch.cuda.stream(copy_in):
                bufs[i]["ind"].copy_(h_ind, non_blocking=True)
                bufs[i]["off"].copy_(h_off, non_blocking=True)
                if h_w is not None:
                    bufs[i]["w"].copy_(h_w, non_blocking=True)
            with torch.cuda.stream(copy_in2):
                bufs[i]["grad"].copy_(h_grad, non_blocking=True)
            copy_in.wait_stream(copy_in2)
            ev_in[i].record(copy_in)

        def e2e_step(k, last):
            i = k % 2
            if not last:
                copy_inputs(1 - i)  # the next step's inputs, while this one computes
            b = bufs[i]
            stream.wait_event(ev_in[i])
            stream.wait_event(ev_out[i])  # the output buffer's previous copy-out is done
            tbe.tbe_forward_prepare(h, b["ind"], b["off"], B, ws, b["w"], b["out"])
            copy_out.wait_stream(stream)
            with torch.cuda.stream(copy_out):
                h_out[i].copy_(b["out"], non_blocking=True)
            ev_out[i].record(copy_out)
            tbe.tbe_backward_apply(h, N, B, b["grad"], ws, cfg.optimizer, cfg.lr, cfg.eps, state)
            ev_used[i].record(stream)

        def e2e_run(steps):
            copy_inputs(0)
            for k in range(steps):
                e2e_step(k, k + 1 == steps)
            stream.wait_stream(copy_out)  # the last output is on the host

        e2e_run(max(1, args.warmup))
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        e_start.record(stream)
        e2e_run(args.steps)
        e_end.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = reduce_max(e_start.elapsed_time(e_end), dev)
        h2d = ind.numel() * ind.element_size() + off.numel() * off.element_size() + \
            (0 if w is None else w.numel() * 4) + grad.numel() * 4
        rec["e2e"] = {"value": units * args.steps / (e2e_ms / 1e3), "unit": "lookups/s", "h2d_bytes_per_step": h2d,
                      "d2h_bytes_per_step": out.numel() * 4, "ms_per_step": e2e_ms / args.steps,
                      "pipelining": "two buffer sets: step k+1's inputs copy in during step k (batch and "
                                    "gradient on two copy streams), step k's output copies out beside its apply",
                      "l2": "not flushed between steps (one timed interval over all steps); the tables "
                            "exceed L2"}
        rc = tbe.tbe_get_error(h)
        if rc != tbe.TBE_OK:
            raise RuntimeError(f"device error in the end-to-end run: {tbe.tbe_strerror(rc)}")
    h.close()
    del tables, batch, grad, ws, out, state, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import recommender_sparse_embeddings_gb300 as tbe

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    extra = [c for c in args.extra if c != args.config]
    with ClockSampler(local) as clk:
        clk.mark_start()
        head = measure(tbe, args.config, args, dev, clk, headline=True)
        others = {str(c): measure(tbe, c, args, dev, clk, headline=False) for c in extra}
        clk.mark_end()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cfg = workloads.get_config(args.config)
        one = cpu_oracle_run(cfg, seconds=args.cpu_seconds, threads=1)
        cores = host_cores()
        allc = cpu_oracle_run(cfg, seconds=args.cpu_seconds, threads=cores, sample=one["oracle_sample"])
        cpu = {"value": allc["lookups"] / allc["seconds"], "unit": "lookups/s", "cores": cores,
               "kind": "oracle", "sample": allc["sample"],
               "one_core": {"value": one["lookups"] / one["seconds"], "cores": 1, "sample": one["sample"]},
               "note": "all host cores: the oracle's OpenMP build of the same source (parallel over bags "
                       "and over runs; the sort is one qsort); one core: the pinned plain build"}

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": head["value"],
            "unit": "lookups/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": head["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": head["dtype"],
            "data": "synthetic: seeded generators with the workload's laws (stand-in for the "
                    "pages' production shard configurations)",
        }
        for k in ("paths", "backward_paths", "config", "fwd", "wgrad", "step_gbs", "segments_ms", "breakdown_ms_sequential",
                  "algorithmic_bytes", "roofline", "ms_per_step_mean", "timed_region_s"):
            line[k] = head[k]
        line["cpu_baseline"] = cpu
        line["e2e"] = head["e2e"]
        line["gpu_launches"] = head["gpu_launches"]
        line["clocks"] = head["clocks"]
        line["clocks_all_workloads"] = clk.summary()
        line["timing"] = ("ms_per_step and every *_ms: median of the K per-step CUDA-event intervals "
                          "(L2 flushed before each step); value = lookups per step / median step time")
        line["workloads"] = {c: {k: v for k, v in r.items() if k not in ("e2e",)} for c, r in others.items()}
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfg = workloads.get_config(args.config)
    # bound the per-step sample so warm-up + timed steps take about two minutes
    # (the oracle does on the order of 1e6 lookups per second per core; the
    # sort stays on one core)
    specs = workloads.realize_tables(cfg)
    per_bag = max(1.0, _mean_bag_length(specs[0]))
    budget_lookups = 120.0 * 1.0e6 / (args.steps + args.warmup)
    bags = int(min(cfg.B, max(64, budget_lookups / per_bag)))
    cores = host_cores()
    sample = OracleSample(cfg, tables_in_sample=1, bags=bags, threads=cores)
    for _ in range(args.warmup):
        sample.step()
    total_s = sum(sample.step() for _ in range(args.steps))
    value = sample.N * args.steps / total_s
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "lookups/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_s / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 accumulate",
        "data": "synthetic: seeded generators with the workload's laws",
        "config": {"workload": cfg.description, "config_id": cfg.cfg_id,
                   "reference": "CPU oracle (plain C, OpenMP build on all host cores); the pages ship no "
                                "implementation to run"},
        "cpu_baseline": {"value": value, "unit": "lookups/s", "cores": cores, "kind": "oracle",
                         "sample": sample.sample + f", {cores} threads"},
        "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", type=int, default=4, help="headline workload")
    p.add_argument("--extra", type=lambda x: [int(c) for c in x.split(",") if c.strip()], default=[2, 3, 5],
                   help="other workloads measured in the same run (comma list; empty: none)")
    p.add_argument("--index-dtype", choices=["int64", "int32"], default="int64")
    p.add_argument("--graph", action="store_true",
                   help="replay the step's two calls as captured CUDA graphs")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-histogram", action="store_true",
                   help="no tensor-core path for small tables (gather forward, sorted backward)")
    p.add_argument("--histogram", choices=["auto", "on", "off"], default="auto",
                   help="small tables' forward on the tensor-core histogram path (TBE_FLAG_FORCE_HISTOGRAM); "
                        "auto: where the workload prescribes it")
    p.add_argument("--length-order", choices=["auto", "on", "off"], default="auto",
                   help="forward bags pooled in order of length (TBE_FLAG_LENGTH_ORDER); auto: for "
                        "workloads whose bag lengths are drawn uniformly over a range spanning 4x or more")
    p.add_argument("--sorted-backward", action="store_true",
                   help="small tables take the sorted backward instead of the dense (tensor-core) one")
    p.add_argument("--tables", type=int, default=0,
                   help="use only the first K tables of the workload (profiling cases)")
    args = p.parse_args(argv)
    args.warmup = max(3, args.warmup)  # timing rule: at least three warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
