"""Decode-step benchmark: TidalDecode PPSA schedule vs the all-full schedule.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--top-k K]
                    [--impl ours|reference] [--no-cpu-baseline]

One "step" is one decode step of the whole L-layer attention-only stack
(full, full+select and sparse layers per the review's Figure 2 schedule) over
one batch of synthetic, seeded inputs resident in HBM.  Default workload: the
largest single-GPU configuration, the long-context LLaMA-2-7B attention shape
(batch 1, 32 layers, 32 heads, d=128, N=102400, k=4096, selection at L2 and
L7; 53.7 GB of K/V resident).  The 10K, 32K and serving shapes run through
--config.

Timing: W untimed warm-up steps, then exactly K timed steps, each preceded by
an L2 flush (a 1 GiB device write, then a 256 MiB read that evicts the
written lines so that their write-back to HBM is over before the step starts;
both outside the timed events), timed with CUDA
events on the launching stream, bracketed by a barrier and a device sync;
the max over ranks is reported.  Pass 1 replays the step as a captured CUDA
graph (the headline latency); pass 2 runs the same K steps through
td_decode_step with per-layer events (per-kernel durations, roofline).
`--impl reference` times the CPU oracle instead (host cores, bounded sample).
Multi-GPU (torchrun): independent replicas, one per GPU, no collective on the
data path (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = ("decode-step attention latency (us) and achieved KV HBM GB/s vs peak, PPSA vs full")
DEFAULT_CONFIG = "llama2-7b-100k"
FLUSH_BYTES = 1 << 30
EVICT_BYTES = 256 << 20  # > the 126 MB L2: a read of it writes back every dirty flush line


class L2Flush:
    """Flush L2 between timed iterations: write FLUSH_BYTES (every line of
    the workload leaves L2), then read EVICT_BYTES of another buffer (the
    dirty lines of the write go back to HBM now, not inside the next timed
    kernel, which would otherwise pay for writing back ~126 MB)."""

    def __init__(self, torch, device):
        self.buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.clean = torch.ones(EVICT_BYTES // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def __call__(self):
        self.buf.fill_(1.0)
        self.sink.copy_(self.clean.sum())

    def describe(self):
        return (f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write, then a "
                f"{EVICT_BYTES >> 20} MiB read that writes the dirty lines back)")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the roofline uses the measured copy peak)


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)


def dist_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity on one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ----------------------------------------------------------------- byte model
def step_bytes(wl: W.Workload, lens: np.ndarray, modes) -> dict:
    """Algorithmic HBM bytes of one step: K/V rows touched (512 B per token per
    KV head at d=128), plus q/out and the index/score traffic listed apart."""
    d, Hkv, Hq, B = wl.head_dim, wl.kv_heads, wl.q_heads, wl.batch
    row = 2 * d * 2                                          # K + V bf16 per token
    full_kv = int(np.sum(lens)) * Hkv * row
    k_eff = np.minimum(lens, wl.top_k)
    sparse_kv = int(np.sum(k_eff)) * Hkv * row
    qo = B * Hq * d * 2 * 2                                  # q read + out write
    per = {"full": full_kv + qo, "sparse": sparse_kv + qo + B * Hkv * wl.top_k * 4}
    kv = {"full": full_kv, "sparse": sparse_kv}
    total_kv = sum(kv["sparse"] if m == W.SPARSE else kv["full"] for m in modes)
    return {"per_launch": per, "kv": kv, "step_kv": total_kv}


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs.

    Samples every `interval_ms`; on entry it waits (at most `first_wait_s`)
    for the first sample, so that the sampler is already running when the
    timed region starts.  The summary counts only samples taken between
    mark_start() and mark_stop() (the whole region when neither is called)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, interval_ms: int = 20, first_wait_s: float = 5.0):
        self.gpu = gpu_index
        self.interval_ms = interval_ms
        self.first_wait_s = first_wait_s
        self.proc = None
        self.lines = []      # (host time, csv line)
        self.t_start = None
        self.t_stop = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < self.first_wait_s:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_start(self):
        self.t_start = time.perf_counter()

    def mark_stop(self):
        self.t_stop = time.perf_counter()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo = self.t_start if self.t_start is not None else -math.inf
        hi = self.t_stop if self.t_stop is not None else math.inf
        for t, ln in self.lines:
            if not lo <= t <= hi:
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "interval_ms": self.interval_ms}


# ----------------------------------------------------------------- oracle timing
HOST_SAMPLE_BYTES = 8 << 30  # host copies of the oracle's sample stay below this


def pick_groups(wl: W.Workload, n_groups: int):
    """Seeded sample of (batch row, KV head) groups for the oracle: at most
    n_groups, and no more than HOST_SAMPLE_BYTES of host K/V copies (a group
    carries every layer's K and V rows)."""
    per_group = wl.layers * wl.max_seq_len * wl.head_dim * 2 * 2
    n_groups = max(1, min(n_groups, HOST_SAMPLE_BYTES // per_group))
    rs = np.random.RandomState(wl.seed + 5)
    all_groups = [(b, g) for b in range(wl.batch) for g in range(wl.kv_heads)]
    n = min(n_groups, len(all_groups))
    return [all_groups[i] for i in sorted(rs.choice(len(all_groups), size=n, replace=False))]


def host_sample(layers, wl: W.Workload, lens, pick):
    """Host copies (bf16 bits) of the sampled groups' q/K/V slices, laid out as
    a batch of len(pick) rows with one KV head each."""
    G = wl.group
    nmax = int(max(lens[b] for b, _ in pick))
    qs, Ks, Vs = [], [], []
    for q, K, V in layers:
        qs.append(np.ascontiguousarray(np.stack([W.u16(q[b, g * G:(g + 1) * G]) for b, g in pick])))
        Ks.append(np.ascontiguousarray(np.stack([W.u16(K[b, g:g + 1, :nmax]) for b, g in pick])))
        Vs.append(np.ascontiguousarray(np.stack([W.u16(V[b, g:g + 1, :nmax]) for b, g in pick])))
    return qs, Ks, Vs, np.array([lens[b] for b, _ in pick], np.int32)


def time_oracle(wl: W.Workload, sample, modes):
    """Seconds the CPU oracle takes for the sample through all layers, and the
    threads it used."""
    import oracle
    orc = oracle.get()
    qs, Ks, Vs, sl = sample
    scale = float(np.float32(1.0) / np.sqrt(np.float32(wl.head_dim)))
    t0 = time.perf_counter()
    _, _, rc = orc.decode_step(list(modes), qs, Ks, Vs, sl, wl.top_k, scale)
    dt = time.perf_counter() - t0
    if rc:
        raise RuntimeError(f"oracle failed: {rc}")
    return dt, orc.num_threads()


# ----------------------------------------------------------------- helpers
def host_cpu_name() -> str:
    """CPU model from /proc/cpuinfo ("model name", else the Arm part number)."""
    try:
        with open("/proc/cpuinfo") as f:
            lines = f.read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "CPU part"):
        for ln in lines:
            if ln.startswith(key):
                return f"{key}: {ln.split(':', 1)[1].strip()}"
    return "unknown"


def load_measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# The sources each attention kernel family is built from: the CUDA-core
# kernels (attention_kernel) and the tensor-core ones (attention_mma*).
ATTN_SOURCES = {"cuda": ("td_attn.cu", "td_attn_common.cuh", "td_internal.h"),
                "mma": ("td_attn_mma.cu", "td_attn_common.cuh", "td_internal.h")}


def kernel_family(kernel: str) -> str:
    return "mma" if kernel.startswith("attention_mma") else "cuda"


def attn_source_hash(family: str) -> str:
    """Hash of one attention kernel family's code (comments and whitespace
    removed, so that an edit to a comment does not retire the DRAM traffic
    ncu measured on the same code)."""
    import re
    h = hashlib.sha256()
    for name in ATTN_SOURCES[family]:
        with open(os.path.join(ROOT, "sparse_attention_td_gb300", "csrc", name)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of one attention kernel ("full" or "sparse") from
    a committed ncu summary, or None if there is none for this workload (name,
    or name-k<top_k> for another k than the workload's own) or the kernel
    source changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(f"{workload}:{kernel}")
    if not entry or entry.get("source_hash") != attn_source_hash(
            kernel_family(entry.get("kernel", ""))):
        return None
    return entry.get("dram_bytes_per_launch")


def consecutive_overlap(td, torch, wl, shape, q, K, V, seq, ws, device):
    """Mean fraction of layer l's top-k set that layer l+1 also selects
    (layers 2..L-1, every (batch row, KV head)), from td_full_attn_select sets
    and td_index_overlap counts; also the Jaccard index of the two sets (both
    of size m = min(k, N_b), sharing c positions: c / (2m - c))."""
    if wl.layers < 4:
        return None
    sets = []
    out = torch.empty_like(q[0])
    for layer in range(2, wl.layers):
        s = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device=device)
        td.td_full_attn_select(shape, q[layer], K[layer], V[layer], seq, wl.top_k, s, out, None,
                               None, ws)
        sets.append(s)
    counts = torch.empty((wl.batch, wl.kv_heads), dtype=torch.int32, device=device)
    size = torch.clamp(seq.to(torch.float32), max=float(wl.top_k)).view(-1, 1)
    rates, jacc = [], []
    for a, b in zip(sets[:-1], sets[1:]):
        td.td_index_overlap(shape, a, b, wl.top_k, counts)
        c = counts.to(torch.float32)
        rates.append((c / size).mean().item())
        jacc.append((c / (2 * size - c)).mean().item())
    return {"mean": round(float(np.mean(rates)), 4), "min": round(float(np.min(rates)), 4),
            "jaccard_mean": round(float(np.mean(jacc)), 4), "layers": f"2..{wl.layers - 1}"}


def coverage_layer(td, torch, wl, shape, q, K, V, seq, ws, device, flush_l2, stream,
                   tau=0.1, reps=20):
    """One selection layer (layer 2) with a coverage budget (tau, at most top_k
    positions) against the same layer with top-k: launch times (events, L2
    flushed before each launch) and the mean budget chosen."""
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device=device)
    counts = torch.empty((wl.batch, wl.kv_heads), dtype=torch.int32, device=device)
    out = torch.empty_like(q[2])

    def timed(fn):
        ev = []
        for i in range(reps + 3):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if i >= 3:
                ev.append((a, b))
        torch.cuda.synchronize(device)
        return statistics.fmean(a.elapsed_time(b) for a, b in ev) * 1e3

    t_cov = timed(lambda: td.td_full_attn_select_coverage(
        shape, q[2], K[2], V[2], seq, tau, wl.top_k, idx, counts, out, None, None, ws,
        stream=stream))
    t_topk = timed(lambda: td.td_full_attn_select(shape, q[2], K[2], V[2], seq, wl.top_k, idx, out,
                                                  None, None, ws, stream=stream))
    return {"tau": tau, "k_max": wl.top_k, "layer_us": round(t_cov, 2),
            "top_k_layer_us": round(t_topk, 2),
            "mean_budget": round(float(counts.to(torch.float32).mean().item()), 1)}


# ----------------------------------------------------------------- our arm
def apply_tuning(td, pairs):
    for kv in pairs:
        key, _, value = kv.partition("=")
        td.td_set_tuning(key, int(value))


def run_ours(args, world, rank, local):
    import torch
    import sparse_attention_td_gb300 as td
    if not os.path.exists(td.lib_path()):
        import __graft_entry__
        __graft_entry__.build()
    apply_tuning(td, args.tuning)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")

    wl = W.WORKLOADS[args.config]
    if args.top_k:
        wl = wl.with_(top_k=args.top_k)
    heavy = W.heavy_positions(wl)
    lens = W.seq_lens(wl)
    layers = [W.generate_layer(wl, layer, device, heavy[layer]) for layer in range(wl.layers)]
    # every layer's q (and output) is a slice of one buffer
    q_all = torch.stack([x[0] for x in layers])
    q = list(q_all.unbind(0))
    K = [x[1] for x in layers]
    V = [x[2] for x in layers]
    seq = torch.as_tensor(lens).to(device)
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                          scale=td.default_scale(wl.head_dim))
    outs_all = torch.empty_like(q_all)
    outs = list(outs_all.unbind(0))
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device=device)
    ws = td.Workspace(shape, wl.top_k, device=device)
    modes = list(wl.modes)
    full_modes = list(W.all_full_schedule(wl.layers))
    sel_modes = list(W.per_layer_select_schedule(wl.layers))
    plan = td.Plan(shape, modes, q, K, V, seq, wl.top_k, idx, outs, None, ws)
    plan_full = td.Plan(shape, full_modes, q, K, V, seq, wl.top_k, idx, outs, None, ws)
    plan_sel = td.Plan(shape, sel_modes, q, K, V, seq, wl.top_k, idx, outs, None, ws)
    # the same step without its sparse layers: the PPSA step minus this one is
    # what the sparse layers cost inside the graph step (their overlap with
    # neighbouring layers included, which per-layer events would break)
    dense = [i for i, m in enumerate(modes) if m != W.SPARSE]
    plan_dense = td.Plan(shape, [modes[i] for i in dense], [q[i] for i in dense],
                         [K[i] for i in dense], [V[i] for i in dense], seq, wl.top_k, idx,
                         [outs[i] for i in dense], None, ws)
    # the same PPSA step with the new token's K/V rows appended to every layer's
    # cache by the attention kernels themselves (rewrites position N_b - 1)
    gen = torch.Generator(device=device).manual_seed(wl.seed + 77)
    k_new = [torch.randn(wl.batch, wl.kv_heads, wl.head_dim, generator=gen, device=device)
             .to(torch.bfloat16) for _ in range(wl.layers)]
    v_new = [torch.randn(wl.batch, wl.kv_heads, wl.head_dim, generator=gen, device=device)
             .to(torch.bfloat16) for _ in range(wl.layers)]
    plan_app = td.Plan(shape, modes, q, K, V, seq, wl.top_k, idx, outs, None, ws,
                       k_new=k_new, v_new=v_new)
    flush_l2 = L2Flush(torch, device)
    sink = torch.zeros(4096, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    K_steps, W_steps = args.steps, args.warmup

    def graph_pass(p, n):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            flush_l2()
            a.record(stream)
            p.launch(stream)
            b.record(stream)
        return ev

    # warm-up
    for _ in range(W_steps):
        flush_l2()
        plan.launch(stream)
        flush_l2()
        plan_full.launch(stream)
        flush_l2()
        plan_sel.launch(stream)
        flush_l2()
        plan_app.launch(stream)
        flush_l2()
        plan_dense.launch(stream)
        td.td_decode_step(shape, modes, q, K, V, seq, wl.top_k, idx, outs, None, ws,
                          stream=stream)
    torch.cuda.synchronize(device)

    # pass 1: the step as a graph (headline), then the all-full schedule
    with ClockSampler(local) as clocks:
        dist_barrier(world, device)
        torch.cuda.synchronize(device)
        clocks.mark_start()
        t_wall = time.perf_counter()
        ev_ppsa = graph_pass(plan, K_steps)
        torch.cuda.synchronize(device)
        wall_ppsa = time.perf_counter() - t_wall
        dist_barrier(world, device)
        ev_full = graph_pass(plan_full, K_steps)
        torch.cuda.synchronize(device)
        dist_barrier(world, device)
        ev_sel = graph_pass(plan_sel, K_steps)
        torch.cuda.synchronize(device)
        dist_barrier(world, device)
        ev_app = graph_pass(plan_app, K_steps)
        torch.cuda.synchronize(device)
        dist_barrier(world, device)
        ev_dense = graph_pass(plan_dense, K_steps)
        torch.cuda.synchronize(device)
        dist_barrier(world, device)
        # pass 2: per-layer events around each layer's launches
        traced = []
        probe = []
        for _ in range(K_steps):
            flush_l2()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(wl.layers + 1)]
            td.td_decode_step(shape, modes, q, K, V, seq, wl.top_k, idx, outs, None, ws,
                              stream=stream, layer_events=e)
            traced.append(e)
        # pass 3: the same layers with only their K/V reads (the read probe), same
        # launch shapes: the memory-system floor of each layer's access pattern
        for _ in range(K_steps):
            flush_l2()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(wl.layers + 1)]
            for layer, m in enumerate(modes):
                e[layer].record(stream)
                td.td_probe_layer_reads(shape, K[layer], V[layer], seq,
                                        idx if m == W.SPARSE else None, wl.top_k, sink,
                                        stream=stream)
            e[wl.layers].record(stream)
            probe.append(e)
        torch.cuda.synchronize(device)
        clocks.mark_stop()
        dist_barrier(world, device)
    ppsa_us = statistics.fmean(a.elapsed_time(b) for a, b in ev_ppsa) * 1e3
    full_us = statistics.fmean(a.elapsed_time(b) for a, b in ev_full) * 1e3
    sel_us = statistics.fmean(a.elapsed_time(b) for a, b in ev_sel) * 1e3
    app_us = statistics.fmean(a.elapsed_time(b) for a, b in ev_app) * 1e3
    dense_us = statistics.fmean(a.elapsed_time(b) for a, b in ev_dense) * 1e3
    per_layer = np.array([[e[i].elapsed_time(e[i + 1]) * 1e3 for i in range(wl.layers)]
                          for e in traced])                      # [K, L] us
    traced_step_us = float(np.mean([e[0].elapsed_time(e[-1]) * 1e3 for e in traced]))
    layer_mean = per_layer.mean(axis=0)
    probe_mean = np.array([[e[i].elapsed_time(e[i + 1]) * 1e3 for i in range(wl.layers)]
                           for e in probe]).mean(axis=0)
    by_mode, floor_by_mode = {}, {}
    for name, m in (("full", W.FULL), ("full_select", W.FULL_SELECT), ("sparse", W.SPARSE)):
        sel = [i for i, mm in enumerate(modes) if mm == m]
        if sel:
            by_mode[name] = float(np.mean(layer_mean[sel]))
            floor_by_mode[name] = float(np.mean(probe_mean[sel]))
    ppsa_us = dist_max(ppsa_us, world, device)
    full_us = dist_max(full_us, world, device)
    sel_us = dist_max(sel_us, world, device)
    app_us = dist_max(app_us, world, device)
    dense_us = dist_max(dense_us, world, device)

    # Figure 4(a)'s measure on this data (untimed): the top-k set each layer
    # would select, and its overlap with the next layer's
    overlap = consecutive_overlap(td, torch, wl, shape, q, K, V, seq, ws, device)
    coverage = coverage_layer(td, torch, wl, shape, q, K, V, seq, ws, device, flush_l2, stream)

    # e2e through the library's host-buffer plan (td_plan_create_host): every
    # step copies each layer's q rows in from page-locked host memory and its
    # output back; the step is complete, outputs on the host, when b fires
    q_host = q_all.cpu().pin_memory()
    o_host = torch.empty(outs_all.shape, dtype=outs_all.dtype).pin_memory()
    h2d = q_host.numel() * q_host.element_size()
    d2h = o_host.numel() * o_host.element_size()
    plan_host = td.Plan(shape, modes, q, K, V, seq, wl.top_k, idx, outs, None, ws,
                        q_host=q_host, out_host=o_host)
    for _ in range(max(W_steps, 1)):
        plan_host.launch(stream)
    torch.cuda.synchronize(device)
    dist_barrier(world, device)
    e2e_ev = []
    for _ in range(K_steps):
        flush_l2()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan_host.launch(stream)
        b.record(stream)
        e2e_ev.append((a, b))
    torch.cuda.synchronize(device)
    assert torch.equal(o_host.to(device), outs_all), "host outputs differ from the device step's"
    plan_host.close()
    e2e_us = dist_max(statistics.fmean(a.elapsed_time(b) for a, b in e2e_ev) * 1e3, world, device)
    assert ws.status() == 0, "device status word set during the bench"

    bytes_model = step_bytes(wl, lens, modes)
    peaks, peak_kind = load_measured_peaks()
    peak = float(peaks["hbm_gbs"])
    # Roofline of each attention kernel from the traced pass: algorithmic bytes
    # of one launch / its mean layer time.  The full kernel's launches are the
    # full layers (full+select layers add the top-k kernel to the layer time).
    # The step's dominant kernel is the one with the most time in the step.
    counts = {name: sum(1 for m in modes if m == mm)
              for name, mm in (("full", W.FULL), ("full_select", W.FULL_SELECT),
                               ("sparse", W.SPARSE))}
    step_sum = sum(by_mode[k] * counts[k] for k in by_mode)
    kernels = {}
    full_launch_us = by_mode.get("full", by_mode.get("full_select"))
    kernels["full"] = {
        "kernel": td.td_kernel_name(shape, 0, False)
                  + ": split-K flash decode over all N_b tokens + combine",
        "launch_us": full_launch_us, "bytes": bytes_model["per_launch"]["full"],
        "floor_us": floor_by_mode.get("full", floor_by_mode.get("full_select")),
        "share": (full_launch_us * (counts["full"] + counts["full_select"])) / step_sum}
    if "sparse" in by_mode:
        kernels["sparse"] = {
            "kernel": td.td_kernel_name(shape, wl.top_k, True)
                      + ": gather of the k persisted K/V rows + combine",
            "launch_us": by_mode["sparse"], "bytes": bytes_model["per_launch"]["sparse"],
            "floor_us": floor_by_mode["sparse"],
            "share": by_mode["sparse"] * counts["sparse"] / step_sum}
    rooflines = {}
    # ncu summaries are keyed by workload, and by k where it is not the workload's own
    traffic_key = wl.name if wl.top_k == W.WORKLOADS[wl.name].top_k else f"{wl.name}-k{wl.top_k}"
    for name, kk in kernels.items():
        ach = kk["bytes"] / (kk["launch_us"] * 1e-6) / 1e9
        rooflines[name] = {
            "kernel": kk["kernel"], "bound": "hbm", "achieved": round(ach, 1), "peak": peak,
            "unit": "GB/s", "frac": round(ach / peak, 4),
            "frac_of_nominal": round(ach / NOMINAL_HBM_GBS, 4),
            "traffic": measured_traffic(traffic_key, name), "peak_source": f"{peak_kind} hbm_gbs",
            "algorithmic_bytes_per_launch": kk["bytes"], "launch_us": round(kk["launch_us"], 2),
            "read_floor_us": round(kk["floor_us"], 2),
            "frac_of_read_floor": round(kk["floor_us"] / kk["launch_us"], 4),
            "share_of_traced_step": round(kk["share"], 4)}
    dominant = max(kernels, key=lambda k: kernels[k]["share"])
    sparse_gbs = rooflines["sparse"]["achieved"] if "sparse" in rooflines else None
    launches_per_step = sum(2 if m == W.FULL_SELECT else 1 for m in modes)
    # the sparse layers inside the graph step: PPSA step minus the same step
    # without them, against the K/V bytes they read
    n_sparse = counts["sparse"]
    sparse_phase = None
    if n_sparse:
        phase_us = ppsa_us - dense_us
        phase_gbs = n_sparse * bytes_model["per_launch"]["sparse"] / (phase_us * 1e-6) / 1e9
        sparse_phase = {
            "dense_step_us": round(dense_us, 2), "sparse_layers": n_sparse,
            "phase_us": round(phase_us, 2), "per_layer_us": round(phase_us / n_sparse, 2),
            "achieved": round(phase_gbs, 1), "unit": "GB/s", "frac": round(phase_gbs / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs",
            "what": "graph step minus the same graph without its sparse layers; bytes = the "
                    "sparse layers' algorithmic bytes (K/V rows, indices, q, out)"}

    result = None
    if rank == 0:
        result = {
            "metric": METRIC,
            "value": round(ppsa_us, 2),
            "unit": "us",
            "n_gpus": world,
            "steps": K_steps,
            "warmup": W_steps,
            "ms_per_step": round(ppsa_us / 1e3, 5),
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 K/V/q with planted heavy positions)",
            "config": {
                "workload": wl.name, "batch": wl.batch, "layers": wl.layers,
                "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "head_dim": wl.head_dim,
                "seq_len": wl.max_seq_len, "seq_len_sum": int(np.sum(lens)), "top_k": wl.top_k,
                "schedule": "".join("FSP"[m] for m in modes),
                "l2": flush_l2.describe(),
                "parallelism": f"replicas x{world}",
                "timing": "CUDA-graph step, CUDA events on the launching stream, mean of K",
            },
            "kv_bytes_per_step": bytes_model["step_kv"],
            "kv_gbs": round(bytes_model["step_kv"] / (ppsa_us * 1e-6) / 1e9, 1),
            "kv_frac_of_peak": round(bytes_model["step_kv"] / (ppsa_us * 1e-6) / 1e9 / peak, 4),
            "all_full_us": round(full_us, 2),
            "all_full_kv_gbs": round(bytes_model["kv"]["full"] * wl.layers / (full_us * 1e-6) / 1e9,
                                     1),
            "speedup_vs_all_full": round(full_us / ppsa_us, 3),
            "per_layer_select_us": round(sel_us, 2),
            "speedup_vs_per_layer_select": round(sel_us / ppsa_us, 3),
            "consecutive_layer_overlap": overlap,
            "append_step_us": round(app_us, 2),
            "coverage_selection": coverage,
            "traced_step_us": round(traced_step_us, 2),
            "layer_us": {k: round(v, 2) for k, v in by_mode.items()},
            "sparse_layer_gbs": round(sparse_gbs, 1) if sparse_gbs else None,
            "sparse_phase_in_graph": sparse_phase,
            "roofline": rooflines[dominant],
            "rooflines": rooflines,
            "gpu_launches": launches_per_step * K_steps,
            "e2e": {"value": round(e2e_us, 2), "unit": "us", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "copies": "inside the captured step: copy kernels over the chip-to-chip "
                              "link in the launch chain (q before layer 0, the last two "
                              "layers' outputs after the last) and copy-engine copies on a "
                              "second stream (the other outputs, every 8 layers; q rows "
                              "beyond 1 MiB beside layer 0)"},
            "clocks": clocks.summary(),
            "wall_s_pass1": round(wall_ppsa, 3),
        }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        pick = pick_groups(wl, args.cpu_groups)
        sample = host_sample(layers, wl, lens, pick)
        groups = wl.batch * wl.kv_heads
        secs, threads, reps = 0.0, 1, 0
        while secs < args.cpu_seconds and reps < 50:
            dt, threads = time_oracle(wl, sample, modes)
            secs += dt
            reps += 1
        per_step_us = secs / reps * (groups / len(pick)) * 1e6
        result["cpu_baseline"] = {
            "value": round(per_step_us, 1), "unit": "us", "cores": min(threads, len(pick)),
            "kind": "oracle",
            "sample": f"{len(pick)} of {groups} (batch row, KV head) groups through all "
                      f"{wl.layers} layers, x{reps} runs, scaled to the whole step",
        }
        # the same oracle on one thread, on a smaller sample (same scaling)
        import oracle
        orc = oracle.get()
        one = pick[:max(1, len(pick) // 8)]
        sample1 = host_sample(layers, wl, lens, one)
        orc.set_threads(1)
        try:
            dt1, _ = time_oracle(wl, sample1, modes)
        finally:
            orc.set_threads(threads)
        result["cpu_baseline"].update({
            "value_1_thread": round(dt1 * (groups / len(one)) * 1e6, 1),
            "sample_1_thread": f"{len(one)} of {groups} groups, one run, scaled",
            "host_cpus": os.cpu_count(), "host_cpu": host_cpu_name()})
    return result


# ----------------------------------------------------------------- reference arm
def run_reference(args, world, rank, local):
    if rank != 0:
        return None
    import torch
    wl = W.WORKLOADS[args.config]
    if args.top_k:
        wl = wl.with_(top_k=args.top_k)
    heavy = W.heavy_positions(wl)
    lens = W.seq_lens(wl)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layers = [W.generate_layer(wl, layer, dev, heavy[layer]) for layer in range(wl.layers)]
    pick = pick_groups(wl, args.cpu_groups)
    sample = host_sample(layers, wl, lens, pick)
    n_done = len(pick)
    del layers
    groups = wl.batch * wl.kv_heads
    times, threads = [], 1
    for i in range(args.warmup + args.steps):
        dt, threads = time_oracle(wl, sample, wl.modes)
        if i >= args.warmup:
            times.append(dt * (groups / n_done) * 1e6)
    value = statistics.fmean(times)
    sample = (f"{n_done} of {groups} (batch row, KV head) groups through all {wl.layers} layers "
              f"per step, scaled to the whole step")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.batch, "layers": wl.layers,
                   "q_heads": wl.q_heads, "kv_heads": wl.kv_heads, "seq_len": wl.max_seq_len,
                   "top_k": wl.top_k, "parallelism": "host cores (oracle)"},
        "cpu_baseline": {"value": round(value, 1), "unit": "us", "cores": min(threads, n_done),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_profile_layer(args, local):
    """One layer of the workload, launched alone W + K times with an L2 flush
    before each launch: the small case for ncu captures (one layer resident)."""
    import torch
    import sparse_attention_td_gb300 as td
    if not os.path.exists(td.lib_path()):
        import __graft_entry__
        __graft_entry__.build()
    apply_tuning(td, args.tuning)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    wl = W.WORKLOADS[args.config]
    if args.top_k:
        wl = wl.with_(top_k=args.top_k)
    layer = 2  # a selection layer of every 32-layer schedule
    heavy = W.heavy_positions(wl)[layer]
    lens = W.seq_lens(wl)
    q, K, V = W.generate_layer(wl, layer, device, heavy)
    seq = torch.as_tensor(lens).to(device)
    shape = td.make_shape(wl.batch, wl.q_heads, wl.kv_heads, wl.max_seq_len,
                          scale=td.default_scale(wl.head_dim))
    out = torch.empty_like(q)
    idx = torch.full((wl.batch, wl.kv_heads, wl.top_k), -1, dtype=torch.int32, device=device)
    ws = td.Workspace(shape, wl.top_k, device=device)
    td.td_full_attn_select(shape, q, K, V, seq, wl.top_k, idx, out, None, None, ws)
    flush = L2Flush(torch, device)

    def op():
        if args.profile == "full":
            td.td_full_attn_select(shape, q, K, V, seq, 0, None, out, None, None, ws)
        elif args.profile == "select":
            td.td_full_attn_select(shape, q, K, V, seq, wl.top_k, idx, out, None, None, ws)
        else:
            td.td_sparse_attn(shape, q, K, V, seq, idx, wl.top_k, out, None, ws)

    times = []
    for i in range(args.warmup + args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        op()
        b.record()
        if i >= args.warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    us = statistics.fmean(a.elapsed_time(b) for a, b in times) * 1e3
    bm = step_bytes(wl, lens, [W.FULL])
    nbytes = bm["per_launch"]["sparse" if args.profile == "sparse" else "full"]
    assert ws.status() == 0
    return {"profile": args.profile, "workload": wl.name, "top_k": wl.top_k, "launch_us": round(us, 2),
            "algorithmic_bytes": nbytes, "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
            "splits": td.td_query_splits(shape, wl.top_k, args.profile == "sparse")}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(W.WORKLOADS))
    ap.add_argument("--top-k", type=int, default=0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-groups", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", choices=["full", "select", "sparse"], default=None,
                    help="time one layer's launch alone (small case for ncu)")
    ap.add_argument("--tuning", action="append", default=[], metavar="KEY=VALUE",
                    help="td_set_tuning before running (repeatable), e.g. mma=0")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.profile:
        res = run_profile_layer(args, local)
    elif args.impl == "reference":
        res = run_reference(args, world, rank, local)
    else:
        res = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
