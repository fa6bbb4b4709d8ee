"""Benchmark of the fused sharded optimizer step on GB300.

Default workload: the GPT-2-Large-shaped ZeRO-1 step (N = 8 simulated ranks,
38 units, Psi = 774,030,080 parameters, bf16 gradients, fp32 master/m/v, bf16
gathered params).  One step = one zero_step call = reduce-scatter + average +
AdamW + bf16 cast + all-gather over every unit, one kernel launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

Prints one JSON line (rank 0).  value = parameters updated per second over
all GPUs (each GPU runs its own full simulated-N-rank step: weak scaling);
e2e = the same metric with the step's gradients copied in from pinned host
memory and the gathered params copied back, every step; roofline = the fused
kernel's algorithmic bytes / its CUDA-event duration against the measured HBM
copy peak; cpu_baseline = the CPU oracle, single-threaded, on a bounded sample.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded-step params/sec and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = [os.path.join(ROOT, "fsdp_sharded_optimizer_step_gb300", "csrc", f)
              for f in ("zero_kernels.cu", "zero_launch.h", "zero_internal.h")]


def kernel_source_hash():
    """First 16 hex digits of the SHA-256 of the kernels' source and the structs they use."""
    h = hashlib.sha256()
    for path in KERNEL_SRC:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(workload, kind="fused"):
    """DRAM bytes (read + write) of one step's update launch(es) from the committed
    ncu summary (kind "fused": the one fused launch; "clip": reduce + finalize +
    shard), or None when the summary is missing or the kernel changed since."""
    return _summary_traffic(f"k_pipe_{kind}_{workload}.md", kernel_source_hash())


def _summary_traffic(name, source_hash):
    try:
        text = open(os.path.join(ROOT, "profiles", name)).read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m or not t or m.group(1) != source_hash:
        return None
    return int(t.group(1))


def reshard_source_hash():
    """First 16 hex digits of the SHA-256 of the reshard kernel's source and the structs it uses."""
    h = hashlib.sha256()
    for f in ("zero_reshard.cu", "zero_internal.h"):
        with open(os.path.join(ROOT, "fsdp_sharded_optimizer_step_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.samples = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        self.mark = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.6)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def begin(self):
        self.mark = time.time()

    def end(self):
        self.mark_end = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [p for (t, p) in self.samples if self.mark is not None and self.mark - 0.2 <= t <= self.mark_end + 0.2]
        use = inside if inside else [p for (_, p) in self.samples]
        if not use:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        mx = [num(p[2]) for p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in use for i in range(4) if p[5 + i].lower().startswith("active")})
        pw = [num(p[3]) for p in use if num(p[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "sm_mhz_min": min(sm) if sm else None, "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------------ distributed plumbing
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        from datetime import timedelta
        backend = "nccl" if torch.cuda.is_available() and args.impl != "reference" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        # a rank that dies or never arrives makes the others' next collective fail after
        # dist_timeout seconds instead of hanging (the ranks share no device work)
        dist.init_process_group(backend=backend, timeout=timedelta(seconds=args.dist_timeout))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """Largest value of x over all ranks (float)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle (baseline only)
def oracle_sample_rate(cfg, n_elems, min_seconds, seed=7, max_steps=1000):
    """The CPU oracle as it stands (single-threaded C), timed on host cores over a
    bounded sample of the workload: one unsharded step over n_elems positions,
    repeated until min_seconds have passed.  Returns (params/s, steps, seconds)."""
    from oracle import oracle as O
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    N = cfg["N"]
    g = W.make_grads(N, n_elems, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device="cpu", seed=seed)
    rows = ([r for r in g.view(torch.int16).numpy().view(np.uint16)] if cfg["gdtype"] == W.BF16
            else [r for r in g.numpy()])
    w = (torch.randn(n_elems, generator=torch.Generator().manual_seed(seed)) * 0.02).numpy()
    m = np.zeros(n_elems, np.float32)
    v = np.zeros(n_elems, np.float32)
    pd = O.BF16 if cfg["pdtype"] == W.BF16 else O.F32
    gd = O.BF16 if cfg["gdtype"] == W.BF16 else O.F32
    steps, t0 = 0, time.perf_counter()
    while True:
        hp = O.hparams(t=steps + 1, max_norm=cfg.get("max_norm", 0.0))
        O.step(rows, gd, w, m, v, hp, pdtype=pd)
        steps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or steps >= max_steps:
            return n_elems * steps / el, steps, el


def oracle_step_all_cores(ex, n_chunks, rows, gd, w, m, v, hp, pd, max_norm):
    """One oracle step over all positions, split into n_chunks contiguous chunks run
    on the threads of `ex`: the oracle's own functions on each chunk (the update is
    element-wise; the clip's exact sums of squares are merged exactly), so w, m, v,
    the output and S are bit-identical to one single-threaded oracle step.
    Returns (status, output, S)."""
    from oracle import oracle as O
    n = w.size
    cuts = [n * k // n_chunks for k in range(n_chunks + 1)]
    parts = [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    coef, S = 1.0, float("nan")
    if max_norm > 0:
        def partial(ab):
            acc = O.SqAcc()
            acc.add_avg_grad([r[ab[0]:ab[1]] for r in rows], gd)
            return acc
        accs = list(ex.map(partial, parts))
        for acc in accs[1:]:
            accs[0].merge(acc)
        S = accs[0].result() if accs else 0.0
        coef = O.clip_coef(S, max_norm)
        if np.isnan(coef):
            return O.ENONFINITE, None, S
    outs = list(ex.map(lambda ab: O.adamw([r[ab[0]:ab[1]] for r in rows], gd, w[ab[0]:ab[1]], m[ab[0]:ab[1]],
                                          v[ab[0]:ab[1]], hp, pdtype=pd, clip=max_norm > 0, coef=coef), parts))
    return O.OK, np.concatenate(outs) if outs else np.zeros(0), S


def oracle_all_cores_rate(cfg, n_elems, min_seconds, seed=7, max_steps=2000):
    """The same sample as oracle_sample_rate, each step run by oracle_step_all_cores on
    every host thread this process may use.  Returns (params/s, steps, seconds, threads)."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import oracle as O
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    N = cfg["N"]
    g = W.make_grads(N, n_elems, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device="cpu", seed=seed)
    rows = ([r for r in g.view(torch.int16).numpy().view(np.uint16)] if cfg["gdtype"] == W.BF16
            else [r for r in g.numpy()])
    w = (torch.randn(n_elems, generator=torch.Generator().manual_seed(seed)) * 0.02).numpy()
    m = np.zeros(n_elems, np.float32)
    v = np.zeros(n_elems, np.float32)
    pd = O.BF16 if cfg["pdtype"] == W.BF16 else O.F32
    gd = O.BF16 if cfg["gdtype"] == W.BF16 else O.F32
    threads = len(os.sched_getaffinity(0))
    max_norm = cfg.get("max_norm", 0.0)
    with ThreadPoolExecutor(threads) as ex:
        steps, t0 = 0, time.perf_counter()
        while True:
            hp = O.hparams(t=steps + 1, max_norm=max_norm)
            oracle_step_all_cores(ex, threads, rows, gd, w, m, v, hp, pd, max_norm)
            steps += 1
            el = time.perf_counter() - t0
            if el >= min_seconds or steps >= max_steps:
                return n_elems * steps / el, steps, el, threads


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this workload."""
    if rank != 0:
        return 0
    from oracle import build as obuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    obuild.build()
    cfg = W.CONFIGS[args.config]
    n = args.ref_sample
    from oracle import oracle as O
    N = cfg["N"]
    g = W.make_grads(N, n, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device="cpu", seed=7)
    rows = ([r for r in g.view(torch.int16).numpy().view(np.uint16)] if cfg["gdtype"] == W.BF16
            else [r for r in g.numpy()])
    w = (torch.randn(n, generator=torch.Generator().manual_seed(7)) * 0.02).numpy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    pd = O.BF16 if cfg["pdtype"] == W.BF16 else O.F32
    gd = O.BF16 if cfg["gdtype"] == W.BF16 else O.F32
    for s in range(args.warmup):
        O.step(rows, gd, w, m, v, O.hparams(t=s + 1, max_norm=cfg.get("max_norm", 0.0)), pdtype=pd)
    t0 = time.perf_counter()
    for s in range(args.steps):
        O.step(rows, gd, w, m, v, O.hparams(t=args.warmup + s + 1, max_norm=cfg.get("max_norm", 0.0)), pdtype=pd)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    sample = f"{n} positions of the {args.config} workload (N={N} ranks), one unsharded oracle step per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": workload_config(args.config, cfg, None),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(name, cfg, plan):
    units = cfg["units"]()
    d = {"workload": f"{name}: {cfg['desc']}", "sim_ranks": cfg["N"], "units": len(units), "psi": int(sum(units)),
         "grad_dtype": cfg["gdtype"], "param_dtype": cfg["pdtype"], "zero_stage": cfg["stage"],
         "clip_max_norm": cfg.get("max_norm", 0.0)}
    if plan is not None:
        d["p_pad"] = plan.P_pad
        if plan.align != 1:
            d["align"] = plan.align
    return d


# ------------------------------------------------------------------ the GPU arm
def update_bytes_per_element(cfg):
    """Algorithmic HBM bytes per padded element of the update launches of one
    step: N gradient reads, master/m/v read and written, one param written (the
    gathered param, or the rank's param shard under ZeRO-3), plus the fp32
    gradient shard written and read back when clipping."""
    gb = 2 if cfg["gdtype"] == "bf16" else 4
    pb = 2 if cfg["pdtype"] == "bf16" else 4
    b = cfg["N"] * gb + 12 + 12 + pb
    if cfg.get("max_norm", 0.0) > 0:
        b += 8
    return b


E2E_PINNED_BUDGET = 32e9


SECONDARY = ("4b_z3", "1p3b_clip", "finewrap", "finewrap600")


def run_secondary(name, steps, warmup, dev):
    """One of the other full-size workloads on this GPU: its whole step timed with CUDA events
    (inputs resident in HBM, larger than L2), the update launch(es) timed on their own, and the
    roofline of each against the measured HBM copy peak.  ZeRO-3 (4b_z3): the fused update writes
    the ranks' param shards (42 B/element) and 33 per-unit all-gathers fill the full buffer
    (4 B/element more: 46 B/element for the whole step)."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    cfg = W.CONFIGS[name]
    sizes = cfg["units"]()
    N = cfg["N"]
    plan = Z.ZeroPlan(sizes, N, dev)
    P, H = plan.P_pad, plan.H
    gdt = torch.bfloat16 if cfg["gdtype"] == W.BF16 else torch.float32
    pdt = torch.bfloat16 if cfg["pdtype"] == W.BF16 else torch.float32
    grads = W.make_grads(N, P, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device=dev, seed=1,
                         outlier_frac=cfg.get("outlier_frac", 0.0), outlier_scale=cfg.get("outlier_scale", 1.0),
                         out=Z.rank_buffers(N, P, gdt, dev))
    master, m, v = W.make_state(N, H, sigma=cfg.get("master_sigma", 0.02), device=dev,
                                out=tuple(Z.rank_buffers(N, H, torch.float32, dev) for _ in range(3)))
    clip = cfg.get("max_norm", 0.0) > 0
    z3 = cfg["stage"] == 3
    full = torch.zeros(P, dtype=pdt, device=dev)
    pshard = Z.rank_buffers(N, H, pdt, dev, zero=True) if z3 else None
    gshard = Z.rank_buffers(N, H, torch.float32, dev) if clip else None
    sq = torch.zeros(1, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(t, ev=None):
        hp = Z.AdamW(t=t, max_norm=cfg.get("max_norm", 0.0), **W.HP)
        if ev is not None:
            ev[0].record(stream)
        Z.zero_step(plan, grads, master, m, v, hp, full=None if z3 else full, pshard=pshard, gshard_ws=gshard,
                    sqnorm_out=sq if clip else None)
        if ev is not None:
            ev[1].record(stream)
        if z3:
            for u in range(plan.n_units):
                Z.zero_all_gather_bf16(plan, pshard, full, unit=u)

    for t in range(1, warmup + 1):
        step(t)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    clocks.start()
    clocks.begin()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        step(warmup + 1 + k, evs[k])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks.end()
    clock_info = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    upd_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    peak, peak_kind = measured_hbm_peak()
    bpe = update_bytes_per_element(cfg)
    upd_gbs = bpe * P / (upd_ms / 1e3) / 1e9
    traffic = ncu_traffic(name, "clip" if clip else "fused")
    out = {"workload": f"{name}: {cfg['desc']}", "psi": int(sum(sizes)), "p_pad": P, "steps": steps, "warmup": warmup,
           "ms_per_step": ms, "params_per_s": int(sum(sizes)) / (ms / 1e3),
           "gpu_launches_per_step": (3 if clip else 1) + (plan.n_units if z3 else 0),
           "update": {"kernel": "k_pipe<REDUCE> + k_finalize + k_pipe<SHARD>" if clip else "k_pipe<FUSED>",
                      "ms": upd_ms, "bytes_per_element": bpe,
                      "roofline": {"bound": "hbm", "achieved": upd_gbs, "peak": peak, "unit": "GB/s",
                                   "frac": upd_gbs / peak, "traffic": traffic, "peak_kind": peak_kind}},
           "clocks": clock_info}
    if name.startswith("finewrap"):
        out["per_unit"] = per_unit_timing(plan, grads, master, m, v, full, steps, warmup, dev, stream, upd_ms)
    step_bpe = bpe + (4 if z3 else 0)  # ZeRO-3: + the per-unit gathers (2 B read + 2 B written per element)
    step_gbs = step_bpe * P / (ms / 1e3) / 1e9
    out["step_roofline"] = {"bound": "hbm", "achieved": step_gbs, "peak": peak, "unit": "GB/s", "frac": step_gbs / peak,
                            "pct_of_8tbs_nominal": 100 * step_gbs / 8000.0, "bytes_per_element": step_bpe,
                            "peak_kind": peak_kind}
    return out


def per_unit_timing(plan, grads, master, m, v, full, steps, warmup, dev, stream, one_launch_ms):
    """The same unclipped step as one launch per unit instead of the one multi-unit launch:
    launched from Python through zero_step, then through UnitSteps (arguments marshalled
    once), then captured in a CUDA graph and replayed (t fixed at capture), each timed
    with CUDA events on the launching stream."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import workloads as W

    def unit_step(t):
        hp = Z.AdamW(t=t, **W.HP)
        for u in range(plan.n_units):
            Z.zero_step(plan, grads, master, m, v, hp, full=full, unit=u)

    def timed(fn, reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    t = 1000
    unit_step(t)
    torch.cuda.synchronize(dev)
    python_ms = timed(lambda: unit_step(t), 1)
    prepared = Z.UnitSteps(plan, grads, master, m, v, full=full)
    hp_t = Z.AdamW(t=t, **W.HP)
    prepared.step(hp_t)
    torch.cuda.synchronize(dev)
    prepared_ms = timed(lambda: prepared.step(hp_t), 1)
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="relaxed"):
        unit_step(t)
    stream.wait_stream(cap)
    torch.cuda.synchronize(dev)
    for _ in range(warmup):
        graph.replay()
    graph_ms = timed(graph.replay, steps)
    del graph
    return {"launches_per_step": plan.n_units, "ms_launched_from_python": python_ms,
            "ms_launched_from_python_marshalled_once": prepared_ms,
            "ms_replayed_from_cuda_graph": graph_ms, "one_launch_ms": one_launch_ms,
            "graph_vs_one_launch": graph_ms / one_launch_ms}


def measure_e2e(args, world, dev, stream, grads, full, step, N, P, gdt, pdt, psi, plan=None, state=None, streamed=False,
                max_norm=0.0, gshard=None):
    """Same metric through the public API with host buffers: every step takes the
    N gradient buffers from pinned host memory and returns the gathered params to
    pinned host memory.  streamed: unit by unit (HostStreamedStep: copy-in of the
    next unit, its update -- or, clipped, its norm pass -- and copy-out of finished
    ones overlap); otherwise all gradients are copied in, the step runs, the params
    are copied out."""
    e2e_steps = max(3, min(args.steps, 10))
    h_grads = torch.empty(N, P, dtype=gdt, pin_memory=True)
    for r in range(N):
        h_grads[r].copy_(grads[r])
    h_full = torch.empty(P, dtype=pdt, pin_memory=True)
    torch.cuda.synchronize(dev)
    if streamed:
        from fsdp_sharded_optimizer_step_gb300 import workloads as W
        from fsdp_sharded_optimizer_step_gb300.binding import AdamW
        from fsdp_sharded_optimizer_step_gb300.streaming import HostStreamedStep
        streamer = HostStreamedStep(plan, gdt)
        master, m, v = state

        def e2e_step(t):
            hp = AdamW(t=t, max_norm=max_norm, **W.HP)
            if max_norm > 0:
                streamer.step_clipped(h_grads, gshard, master, m, v, hp, full, host_full=h_full)
            else:
                streamer.step(h_grads, master, m, v, hp, full, host_full=h_full)
    else:
        def e2e_step(t):
            for r in range(N):
                grads[r].copy_(h_grads[r], non_blocking=True)
            step(t)
            h_full.copy_(full, non_blocking=True)

    for t in range(2):  # warm the copy engines
        e2e_step(10_000 + t)
    torch.cuda.synchronize(dev)
    barrier(world)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps + 1)]
    marks[0].record(stream)
    for k in range(e2e_steps):
        e2e_step(20_000 + k)
        marks[k + 1].record(stream)
    torch.cuda.synchronize(dev)
    per_step = [marks[k].elapsed_time(marks[k + 1]) for k in range(e2e_steps)]
    e2e_ms = max_over_ranks(marks[0].elapsed_time(marks[-1]) / e2e_steps, world, dev)
    h2d = h_grads.numel() * h_grads.element_size()
    d2h = h_full.numel() * h_full.element_size()
    e2e = {"value": world * psi / (e2e_ms / 1e3), "unit": UNIT,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
           # the host link's speed varies from step to step: the per-step spread, and the link rate
           # the fastest step reached (all copied bytes over its time)
           "median_ms": statistics.median(per_step), "min_ms": min(per_step), "max_ms": max(per_step),
           "per_step_ms": [round(x, 2) for x in per_step],
           "link_GBs_at_min": (h2d + d2h) / (min(per_step) / 1e3) / 1e9,
           "mode": ("streamed per unit: copy-in, norm pass, then update and copy-out overlapped" if max_norm > 0
                    else "streamed per unit: copy-in, update and copy-out overlapped") if streamed
           else "copy all gradients in, step, copy params out"}
    del h_grads, h_full
    return e2e


def run_reshard(args, world, rank, local):
    """Checkpoint resharding of the workload's master/m/v from N to N' ranks on the
    device: per step three zero_reshard launches (fp32), 8 bytes of HBM traffic per
    padded element and array (read + write)."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import build as zbuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    zbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    sizes = cfg["units"]()
    N = cfg["N"]
    N2 = args.to_ranks or 2 * N
    pf, pt = Z.ZeroPlan(sizes, N, dev), Z.ZeroPlan(sizes, N2, dev)
    src = W.make_state(N, pf.H, device=dev, out=tuple(Z.rank_buffers(N, pf.H, torch.float32, dev) for _ in range(3)))
    dst = tuple(Z.rank_buffers(N2, pt.H, torch.float32, dev) for _ in range(3))
    stream = torch.cuda.current_stream(dev)

    def step():
        for a, b in zip(src, dst):
            Z.zero_reshard(pf, pt, a, b)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    nbytes = 3 * (pf.H * N * 4 + pt.H * N2 * 4)
    gbs = nbytes / (ms / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    per_launch = _summary_traffic(f"k_reshard_{args.config}_{N}to{N2}.md", reshard_source_hash())
    traffic = None if per_launch is None else 3 * per_launch
    if rank == 0:
        print(json.dumps({"metric": "checkpoint reshard of master/m/v (GB/s of HBM traffic)", "value": world * gbs,
                          "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "f32", "data": "synthetic",
                          "config": {"workload": f"{args.config}: {cfg['desc']}", "from_ranks": N, "to_ranks": N2,
                                     "bytes_per_step": nbytes},
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                       "frac": gbs / peak, "traffic": traffic, "peak_kind": peak_kind,
                                       "per": "step (three launches, one per array)"},
                          "gpu_launches": 3 * args.steps}), flush=True)
    return 0


def run_gather(args, world, rank, local):
    """The all-gather of every unit in one launch (k_gather): bf16 rank shards of the
    workload's layout into the full parameter buffer, 4 bytes of HBM traffic per padded
    element (2 read, 2 written).  Fine-wrap layouts exercise the misaligned path."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import build as zbuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    zbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    sizes = cfg["units"]()
    N = cfg["N"]
    plan = Z.ZeroPlan(sizes, N, dev)
    pshard = Z.rank_buffers(N, plan.H, torch.bfloat16, dev)
    pshard.normal_()
    full = torch.empty(plan.P_pad, dtype=torch.bfloat16, device=dev)
    segs = Z.zero_plan_segments(plan.handle)
    misaligned = sum(1 for sg in segs if (sg[0] - sg[1]) % 8) / max(len(segs), 1)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        Z.zero_all_gather_bf16(plan, pshard, full)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        Z.zero_all_gather_bf16(plan, pshard, full)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    nbytes = 4 * plan.P_pad
    gbs = nbytes / (ms / 1e3) / 1e9
    peak, peak_kind = measured_hbm_peak()
    traffic = _summary_traffic(f"k_gather_{args.config}.md", kernel_source_hash())
    if rank == 0:
        print(json.dumps({"metric": "all-gather of every unit in one launch (GB/s of HBM traffic)", "value": world * gbs,
                          "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                          "dtype": "bf16", "data": "synthetic",
                          "config": {"workload": f"{args.config}: {cfg['desc']}", "bytes_per_step": nbytes,
                                     "segments": len(segs), "misaligned_segment_fraction": misaligned},
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                       "frac": gbs / peak, "traffic": traffic, "peak_kind": peak_kind},
                          "gpu_launches": args.steps}), flush=True)
    return 0


def run_offload(args, world, rank, local):
    """ZeRO-Offload step (zero_offload_step): gradients in HBM, master/m/v in pinned host
    memory, the GPU reduce-scatters batch by batch, the host cores run AdamW as each
    batch's gradient shard lands, the bf16 params go back to HBM.  Reports params/s,
    the host link's rates, the host cores' update rate, and where a step's time goes."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import binding as B
    from fsdp_sharded_optimizer_step_gb300 import build as zbuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    zbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    sizes = cfg["units"]()
    N = cfg["N"]
    plan = Z.ZeroPlan(sizes, N, dev, align=args.align)
    P, H = plan.P_pad, plan.H
    gdt = torch.bfloat16 if cfg["gdtype"] == W.BF16 else torch.float32
    pdt = torch.bfloat16 if cfg["pdtype"] == W.BF16 else torch.float32
    grads = W.make_grads(N, P, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device=dev, seed=1 + 100 * rank,
                         outlier_frac=cfg.get("outlier_frac", 0.0), outlier_scale=cfg.get("outlier_scale", 1.0),
                         out=Z.rank_buffers(N, P, gdt, dev))
    state_dev = W.make_state(N, H, sigma=cfg.get("master_sigma", 0.02), device=dev)
    host = []
    for x in state_dev:
        h = torch.empty(N, H, dtype=torch.float32, pin_memory=True)
        h.copy_(x)
        host.append(h)
    master_h, m_h, v_h = host
    del state_dev
    torch.cuda.empty_cache()
    gshard_dev = Z.rank_buffers(N, H, torch.float32, dev)
    gshard_h = torch.empty(N, H, dtype=torch.float32, pin_memory=True)
    full_h = torch.empty(P, dtype=pdt, pin_memory=True)
    full_dev = torch.empty(P, dtype=pdt, device=dev)
    eng = B.OffloadEngine(plan, n_threads=args.offload_threads, batch_min=args.offload_batch)
    threads, n_batches = Z.zero_offload_info(eng)
    stream = torch.cuda.current_stream(dev)
    max_norm = cfg.get("max_norm", 0.0)

    def step(t):
        hp = Z.AdamW(t=t, max_norm=max_norm, **W.HP)
        rc, _ = Z.zero_offload_step(eng, grads, gshard_dev, gshard_h, master_h, m_h, v_h, full_h, hp,
                                    full_dev=full_dev, stream=stream)
        if rc != B.ZERO_OK:
            raise RuntimeError(f"zero_offload_step returned {rc}")

    for t in range(1, args.warmup + 1):
        step(t)
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    clocks.begin()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.perf_counter()
    e0.record(stream)
    for k in range(args.steps):
        step(args.warmup + 1 + k)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    wall_ms = (time.perf_counter() - w0) * 1e3 / args.steps
    clocks.end()
    clock_info = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    psi = int(sum(sizes))
    # one more step, for the breakdown of where its time goes
    step(args.warmup + args.steps + 1)
    tm = Z.zero_offload_timings(eng)
    # the pieces alone: the host link each way, and the host cores' update
    d2h_bytes, h2d_bytes = 4 * N * H, P * full_h.element_size()

    def copy_ms(dst, src, reps=3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dst.copy_(src, non_blocking=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / reps

    t_d2h = copy_ms(gshard_h, gshard_dev)
    t_h2d = copy_ms(full_dev, full_h)
    hp = Z.AdamW(t=1, **W.HP)
    reps = 3
    Z.zero_offload_adamw(eng, gshard_h, master_h, m_h, v_h, hp, full_h=full_h)
    c0 = time.perf_counter()
    for _ in range(reps):
        Z.zero_offload_adamw(eng, gshard_h, master_h, m_h, v_h, hp, full_h=full_h)
    t_host = (time.perf_counter() - c0) * 1e3 / reps
    host_bytes = N * H * (4 + 12 + 12) + P * full_h.element_size()
    host_peak = host_stream_gbps(threads)
    if rank == 0:
        print(json.dumps({
            "metric": "ZeRO-Offload step params/sec (state in host memory, update on the host cores)",
            "value": world * psi / (ms / 1e3), "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "wall_ms_per_step": wall_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(args.config, cfg, plan), host_threads=threads, batches=n_batches),
            "link": {"d2h_bytes_per_step": d2h_bytes, "h2d_bytes_per_step": h2d_bytes,
                     "d2h_GBps_alone": d2h_bytes / (t_d2h / 1e3) / 1e9, "h2d_GBps_alone": h2d_bytes / (t_h2d / 1e3) / 1e9,
                     "d2h_ms_alone": t_d2h, "h2d_ms_alone": t_h2d},
            "host_update": {"ms_alone": t_host, "params_per_s": psi / (t_host / 1e3),
                            "bytes_per_step": host_bytes, "GBps": host_bytes / (t_host / 1e3) / 1e9,
                            "threads": threads, "host_stream_add_GBps": host_peak,
                            "frac_of_host_stream": host_bytes / (t_host / 1e3) / 1e9 / host_peak},
            "breakdown_one_step_ms": tm,
            "share": {"update_on_cores": tm["update_ms"] / tm["device_to_params_ms"],
                      "waiting_for_link": tm["wait_ms"] / tm["device_to_params_ms"]},
            "gpu_launches": args.steps * (n_batches + (1 if max_norm > 0 else 0)),
            "clocks": clock_info}), flush=True)
    return 0


def host_stream_gbps(threads, n=1 << 28, reps=5):
    """The host's memory bandwidth as a STREAM-style add, z = x + y over three fp32
    arrays of n elements (12 bytes per element) on `threads` torch threads: the
    reference the offloaded update's host traffic is set against."""
    old = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        x, y, z = torch.ones(n), torch.ones(n), torch.empty(n)
        torch.add(x, y, out=z)
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            torch.add(x, y, out=z)
            best = min(best, time.perf_counter() - t0)
        return 12 * n / best / 1e9
    finally:
        torch.set_num_threads(old)


def _time_ms(fn, stream, reps, rounds=3, warm=2):
    """Mean ms per call of fn over reps back-to-back calls (CUDA events on `stream`),
    after `warm` untimed calls; the best of `rounds` such runs."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / reps)
    return best


def run_unit_flows(args, world, rank, local):
    """The steps either side of the update, unit by unit (rank 0 of each GPU reports)."""
    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import build as zbuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    from fsdp_sharded_optimizer_step_gb300.zero3 import BucketedReduceScatter, UnitGatherer
    zbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    sizes = cfg["units"]()
    N = cfg["N"]
    plan = Z.ZeroPlan(sizes, N, dev)
    P, H = plan.P_pad, plan.H
    stream = torch.cuda.current_stream(dev)
    reps = max(args.steps, 1)
    out = {"n_gpus": world, "steps": reps, "warmup": 2, "data": "synthetic",
           "config": {"workload": f"{args.config}: {cfg['desc']}", "units": len(sizes)}}
    clocks = ClockSampler(local)
    clocks.start()
    clocks.begin()
    if args.op == "zero3_gather":
        pshard = Z.rank_buffers(N, H, torch.bfloat16, dev)
        pshard.normal_()
        gatherers = {"kernel": UnitGatherer(plan, pshard)}
        d = 1280
        x = torch.randn(4096, d, dtype=torch.bfloat16, device=dev)
        wmat = torch.randn(d, 4 * d, dtype=torch.bfloat16, device=dev)

        def compute(u, params_u):  # a synthetic per-unit forward: one GEMM
            torch.matmul(x, wmat)

        t_compute = _time_ms(lambda: [compute(u, None) for u in range(plan.n_units)], stream, reps)
        gather_bytes = 2 * P * 2  # bf16 read from the shards + written to the unit buffers
        timeline = {"compute_only_ms": t_compute, "full_param_buffer_bytes": P * 2,
                    "unit_buffers_bytes": sum(b.numel() * b.element_size() for b in gatherers["kernel"].buffers)}
        for e, g in gatherers.items():
            t_pref = _time_ms(lambda: g.run(compute, prefetch=True), stream, reps)
            t_serial = _time_ms(lambda: g.run(compute, prefetch=False), stream, reps)
            t_gather = _time_ms(lambda: g.run(lambda u, p_: None, prefetch=False), stream, reps)
            timeline[e] = {"prefetch_ms": t_pref, "no_prefetch_ms": t_serial, "gather_only_ms": t_gather,
                           "gather_GBps": gather_bytes / (t_gather / 1e3) / 1e9,
                           "hidden_fraction_of_gather": max(0.0, (t_serial - t_pref) / t_gather) if t_gather else None}
        best = min(timeline[e]["prefetch_ms"] for e in gatherers)
        out.update(metric="ZeRO-3 forward timeline: per-unit gather + synthetic GEMM (ms per pass)",
                   value=best, unit="ms", higher_is_better=False, timeline=timeline)
    else:
        from fsdp_sharded_optimizer_step_gb300.zero3 import BucketedStep
        grads = W.make_grads(N, P, W.BF16, device=dev, out=Z.rank_buffers(N, P, torch.bfloat16, dev))
        master, m, v = W.make_state(N, H, device=dev,
                                    out=tuple(Z.rank_buffers(N, H, torch.float32, dev) for _ in range(3)))
        gshard = Z.rank_buffers(N, H, torch.float32, dev)
        full = torch.zeros(P, dtype=torch.bfloat16, device=dev)
        hp = Z.AdamW(t=1, **W.HP)
        t_fused = _time_ms(lambda: Z.zero_step(plan, grads, master, m, v, hp, full=full), stream, reps)

        def fill(u0, u1, view):  # the backward of units [u0, u1): here their gradients already exist
            view.copy_(grads[:, plan.F[u0]:plan.F[u0] + view.shape[1]])

        flows = {}
        state0 = [x.clone() for x in (master, m, v)]
        for label, be in (("one unit per bucket", 1), ("2^26-element buckets", 1 << 26),
                          ("default buckets", None), ("2^28-element buckets", 1 << 28)):
            for x, x0 in zip((master, m, v), state0):  # every flow starts from the same finite state
                x.copy_(x0)
            bs = BucketedStep(plan, bucket_elems=be)
            # every bucket holds real gradients (the first bucket-length positions of each rank):
            # uninitialised memory would feed inf/NaN/subnormal values into the state, and the
            # exact division and square root then take their slow paths in every later launch
            bs.bucket.copy_(grads[:, :bs.bucket.shape[1]])

            def updates():  # the bucket updates alone, back to back (the bucket holds gradients)
                for u0, u1 in bs.buckets:
                    Z.zero_step_units(plan, u0, u1, bs.view(u0, u1), master, m, v, hp, full=full)

            flows[label] = {"buckets": len(bs.buckets), "bucket_bytes": bs.bucket_bytes,
                            "bucket_updates_ms": _time_ms(updates, stream, reps),
                            "total_ms_incl_fill_copies": _time_ms(
                                lambda: bs.step(fill, master, m, v, hp, full=full), stream, reps)}
            del bs
        # the previous flow: per-unit reduce-scatter into the fp32 gradient shard, then the shard update
        for x, x0 in zip((master, m, v), state0):
            x.copy_(x0)
        buckets = BucketedReduceScatter(plan)
        buckets.bucket.copy_(grads[:, :buckets.bucket.shape[1]])
        t_rs = _time_ms(lambda: [Z.zero_reduce_scatter_unit(plan, u, buckets.bucket[:, :plan.S[u]], gshard)
                                 for u in reversed(range(plan.n_units))], stream, reps)
        t_shard = _time_ms(lambda: Z.zero_adamw_shard_step(plan, gshard, master, m, v, hp, full=full), stream, reps)
        t_fused_end = _time_ms(lambda: Z.zero_step(plan, grads, master, m, v, hp, full=full), stream, reps)
        best = flows["default buckets"]["bucket_updates_ms"]
        out.update(metric="ZeRO-2 bucketed step: bucket updates of the default bucketing (ms per step)",
                   value=best, unit="ms", higher_is_better=False,
                   flow={"fused_step_ms": t_fused, "fused_step_ms_at_the_end": t_fused_end, "bucketed": flows,
                         "vs_fused": best / t_fused,
                         "shard_route_ms": {"reduce_scatter_per_unit": t_rs, "shard_update": t_shard},
                         "full_gradient_bytes": N * P * 2, "gradient_shard_bytes": N * H * 4})
    clocks.end()
    out["clocks"] = clocks.stop()
    if rank == 0:
        print(json.dumps(out), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="gpt2l")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--per-unit", action="store_true", help="one launch per unit instead of the multi-unit table")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step's launches in a CUDA graph after the warm-up and replay it in the timed "
                         "region (removes host launch overhead; the step counter t is the one captured)")
    ap.add_argument("--ref-sample", type=int, default=1 << 22)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--align", type=int, default=1,
                    help="pad every unit to a multiple of N*align (slices on align-element boundaries; "
                         "1 = the pages' layout)")
    ap.add_argument("--dist-timeout", type=float, default=300.0,
                    help="seconds a rank waits in a collective (barrier, timing reduction) before it fails")
    ap.add_argument("--secondary", action=argparse.BooleanOptionalAction, default=True,
                    help="with the default gpt2l step on one GPU, also time the 4b_z3, 1p3b_clip and finewrap "
                         "workloads (each after the previous one's buffers are freed) into a 'secondary' block")
    ap.add_argument("--secondary-steps", type=int, default=5)
    ap.add_argument("--offload-threads", type=int, default=0, help="host threads of the offloaded update (0: all)")
    ap.add_argument("--offload-batch", type=int, default=0, help="offload pipeline batch, padded elements (0: 2^22)")
    ap.add_argument("--op", default="step",
                    choices=["step", "reshard", "gather", "zero3_gather", "zero2_buckets", "offload"],
                    help="step: the sharded optimizer step (default); reshard: checkpoint resharding of the state; "
                         "gather: the all-gather of every unit in one launch; "
                         "zero3_gather: per-unit gathers with/without prefetch beside a synthetic per-unit GEMM; "
                         "zero2_buckets: the bucketed ZeRO-2 step against the fused step; "
                         "offload: the ZeRO-Offload step with the state in host memory")
    ap.add_argument("--to-ranks", type=int, default=0, help="reshard target rank count (default 2N)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.op == "reshard":
        return run_reshard(args, world, rank, local)
    if args.op == "gather":
        return run_gather(args, world, rank, local)
    if args.op in ("zero3_gather", "zero2_buckets"):
        return run_unit_flows(args, world, rank, local)
    if args.op == "offload":
        return run_offload(args, world, rank, local)

    import fsdp_sharded_optimizer_step_gb300 as Z
    from fsdp_sharded_optimizer_step_gb300 import build as zbuild
    from fsdp_sharded_optimizer_step_gb300 import workloads as W
    zbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    cfg = W.CONFIGS[args.config]
    sizes = cfg["units"]()
    N = cfg["N"]
    plan = Z.ZeroPlan(sizes, N, dev, align=args.align)
    P, H = plan.P_pad, plan.H
    gdt = torch.bfloat16 if cfg["gdtype"] == W.BF16 else torch.float32
    pdt = torch.bfloat16 if cfg["pdtype"] == W.BF16 else torch.float32
    grads = W.make_grads(N, P, cfg["gdtype"], sigma=cfg.get("grad_sigma", 1e-3), device=dev, seed=1 + 100 * rank,
                         outlier_frac=cfg.get("outlier_frac", 0.0), outlier_scale=cfg.get("outlier_scale", 1.0),
                         out=Z.rank_buffers(N, P, gdt, dev))
    master, m, v = W.make_state(N, H, sigma=cfg.get("master_sigma", 0.02), device=dev,
                                out=tuple(Z.rank_buffers(N, H, torch.float32, dev) for _ in range(3)))
    clip = cfg.get("max_norm", 0.0) > 0
    z3 = cfg["stage"] == 3
    full = torch.zeros(P, dtype=pdt, device=dev)
    pshard = Z.rank_buffers(N, H, pdt, dev, zero=True) if z3 else None
    gshard = Z.rank_buffers(N, H, torch.float32, dev) if clip else None
    sq = torch.zeros(1, dtype=torch.float64, device=dev)
    stream = torch.cuda.current_stream(dev)
    units = list(range(plan.n_units)) if args.per_unit else [-1]

    def step(t, ev=None):
        hp = Z.AdamW(t=t, max_norm=cfg.get("max_norm", 0.0), **W.HP)
        if ev is not None:
            ev[0].record(stream)
        for u in units:
            Z.zero_step(plan, grads, master, m, v, hp, full=None if z3 else full, pshard=pshard,
                        gshard_ws=gshard, sqnorm_out=sq if clip else None, unit=u)
        if ev is not None:
            ev[1].record(stream)
        if z3:
            for u in range(plan.n_units):
                Z.zero_all_gather_bf16(plan, pshard, full, unit=u)

    launches_per_step = len(units) * (3 if clip else 1) + (plan.n_units if z3 else 0)

    for t in range(1, args.warmup + 1):
        step(t)
    torch.cuda.synchronize(dev)
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap, capture_error_mode="relaxed"):
            step(args.warmup + 1)
        stream.wait_stream(cap)
        torch.cuda.synchronize(dev)

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.begin()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        if graph is not None:
            evs[k][0].record(stream)
            graph.replay()
            evs[k][1].record(stream)
        else:
            step(args.warmup + 1 + k, evs[k])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks.end()
    clock_info = clocks.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps
    psi = int(sum(sizes))
    value = world * psi / (ms_per_step / 1e3)

    # the dominant kernel: the update launch(es) of one step, timed on its stream
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    bpe = update_bytes_per_element(cfg)  # the ZeRO-3 gathers run outside these events
    alg_bytes = bpe * P
    peak, peak_kind = measured_hbm_peak()
    achieved = alg_bytes / (kernel_ms / 1e3) / 1e9
    traffic = ncu_traffic(args.config, "clip" if clip else "fused") if not args.per_unit and args.align == 1 else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_kind": peak_kind, "bytes_per_element": bpe,
                "algorithmic_bytes_per_launch": alg_bytes,
                "kernel": "k_pipe<REDUCE> + k_finalize + k_pipe<SHARD>" if clip else "k_pipe<FUSED>"}

    # ---------------- end to end through the public API with host buffers
    pinned_bytes = N * P * grads.element_size() + P * full.element_size()
    if pinned_bytes <= E2E_PINNED_BUDGET:
        e2e = measure_e2e(args, world, dev, stream, grads, full, step, N, P, gdt, pdt, psi, plan=plan,
                          state=(master, m, v), streamed=not (z3 or args.per_unit),
                          max_norm=cfg.get("max_norm", 0.0), gshard=gshard)
    else:
        e2e = {"value": None, "unit": UNIT, "skipped": f"{pinned_bytes / 1e9:.0f} GB of pinned host buffers "
                                                       f"exceeds the {E2E_PINNED_BUDGET / 1e9:.0f} GB budget"}

    # ---------------- the other full-size workloads, each measured after this one's buffers are freed
    secondary = None
    if world == 1 and args.secondary and args.config == "gpt2l" and args.align == 1 and not (args.per_unit or args.graph):
        del step, grads, master, m, v, full, pshard, gshard, sq, graph
        plan = None
        torch.cuda.empty_cache()
        secondary = {}
        for name in SECONDARY:
            secondary[name] = run_secondary(name, args.secondary_steps, 3, dev)
            torch.cuda.empty_cache()

    # ---------------- CPU oracle baseline (rank 0, one GPU only)
    cpu = cpu_all = None
    if rank == 0 and world == 1:
        from oracle import build as obuild
        obuild.build()
        n_cpu = 1 << 23
        rate, nsteps, secs = oracle_sample_rate(cfg, n_cpu, args.cpu_seconds)
        cpu = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"{nsteps} oracle steps over {n_cpu} positions of the {args.config} workload "
                         f"(N={N} ranks), {secs:.1f} s single-threaded"}
        rate, nsteps, secs, threads = oracle_all_cores_rate(cfg, n_cpu, args.cpu_seconds)
        cpu_all = {"value": rate, "unit": UNIT, "cores": threads,
                   "kind": "oracle on all host threads: its functions on one contiguous chunk of positions per "
                           "thread, results bit-identical to the single-threaded oracle",
                   "sample": f"{nsteps} steps over the same {n_cpu} positions, {secs:.1f} s"}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": dict(workload_config(args.config, cfg, plan),
                               l2="inputs larger than L2 (no flush): "
                                  f"{alg_bytes / 1e9:.1f} GB of HBM traffic per step vs 129 MB of L2",
                               launch=("one launch per unit" if args.per_unit else "one multi-unit launch")
                               + (", replayed from one CUDA graph (t fixed at capture)" if args.graph else ""),
                               parallelism=f"{world} GPU(s), each a full replica of the {N}-simulated-rank step"),
                "hbm_gbs": achieved, "pct_of_peak": 100 * achieved / peak,
                "pct_of_8tbs_nominal": 100 * achieved / 8000.0,
                "roofline": roofline, "cpu_baseline": cpu, "cpu_all_cores": cpu_all, "e2e": e2e,
                "secondary": secondary,
                "gpu_launches": args.steps * launches_per_step, "clocks": clock_info,
                "kernel_source_sha256_16": kernel_source_hash(),
                "device": torch.cuda.get_device_name(dev)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
