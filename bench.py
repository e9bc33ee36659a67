#!/usr/bin/env python
"""Benchmark of the attention-KL primitive (forward + backward) on GB300.

One step = streamkl_fwd + streamkl_bwd (both gradient sets) over one batch of
the 64K-context causal workload: B=1, H=32, N_Q=N_K=65536, d=128, bf16,
teacher ~ N(0,1), student = teacher + 0.2 N(0,1), scale = 1/sqrt(128).

Metric: fwd+bwd TFLOP/s at that workload with the usual attention convention,
4 N_Q N_K d (forward) + 8 N_Q N_K d (backward) per head, halved for causal.
The value is device-timed with inputs resident in HBM (inputs are 2 GiB, far
larger than the 129 MB L2, so no flush is needed between steps). ``e2e`` is
the same metric through the public Python API with host (pinned) buffers:
each step copies the inputs in and every result out (KL, LSE1, LSE2 and the
four gradients), the batch streamed in groups of heads: a group's inputs are
copied in on one stream and the previous group's results out on another
while the group in between computes.

``roofline`` counts the method's work: 4d FLOPs per visible (query, key) pair
for the forward, and for the backward 4d to regenerate S1, S2 plus 4d per
gradient set (12d with both sets); what the kernels execute (the separate
dK and dQ kernels each regenerate S1 and S2: 16d) is reported beside it.
``configs`` holds one entry per named workload (times, the same counts, and
the GPU results' error against the oracle on the sample the CPU-baseline leg
times).

``--impl reference`` times the fp64 CPU oracle on the host cores instead (a
bounded sample of the same workload per step).

Under torchrun (N > 1) every rank runs its own replica of the workload on its
own GPU (heads and batches are independent, so there is no exchange step);
the reported time is the maximum over ranks and the value counts all ranks'
work ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "causal64k"
METRIC = "attention-KL fwd+bwd TFLOP/s and ms at 64K causal; % of GB300 BF16 tensor peak"


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-budget-s", type=float, default=15.0,
                   help="target CPU seconds for the oracle sample")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-groups", type=int, default=4,
                   help="(batch, head) groups a step's batch is streamed in for the e2e leg")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the per-workload entries (times and oracle errors)")
    return p.parse_args(argv)


# --------------------------------------------------------------------------- ranks
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=world)
    return rank, world


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a host float over all ranks (identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(rank: int) -> int:
    """Each rank draws its own replica of the workload."""
    return 1000 + rank


# --------------------------------------------------------------------------- work counts
def flop_counts(w):
    """(fwd, bwd_metric) FLOPs for one step in the headline convention:
    4 N_Q N_K d forward and 8 N_Q N_K d backward per head, halved for causal."""
    dense = w.NQ * w.NK * w.d * w.B * w.H
    half = 0.5 if w.causal else 1.0
    return 4 * dense * half, 8 * dense * half


def method_flops(w):
    """(fwd, bwd) FLOPs of the method's work on the exact visible pairs: the
    forward's two score GEMMs (4d per pair); the backward's regeneration of
    S1, S2 (4d) plus dQ_t and dK_t (4d) per gradient set."""
    pairs = w.live_pairs_per_head() * w.B * w.H
    sets = 2 if w.grad1 else 1
    return 4 * pairs * w.d, (4 + 4 * sets) * pairs * w.d


def executed_bwd_flops(w, separate: bool):
    """Backward FLOPs the kernels execute: the separate dK and dQ kernels each
    regenerate S1 and S2, the fused kernel once."""
    pairs = w.live_pairs_per_head() * w.B * w.H
    sets = 2 if w.grad1 else 1
    return ((8 if separate else 4) + 4 * sets) * pairs * w.d


def bwd_min_bytes(w):
    """Bytes the backward must move at least: the four inputs once, the
    gradients it writes once, and the per-row vectors it reads (KL, LSE1,
    LSE2, g)."""
    bh = w.B * w.H
    q = bh * w.NQ * w.d * 2
    k = bh * w.NK * w.d * 2
    sets = 2 if w.grad1 else 1
    return 2 * (q + k) + sets * (q + k) + 4 * bh * w.NQ * 4


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.out.flush()
        self.out.seek(0)
        rows = [r.strip().split(",") for r in self.out.read().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                r = [x.strip() for x in r]
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                power.append(float(r[3]))
                for n, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p >= 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- CPU oracle
def draw_head(w, seed: int = 7):
    """One (batch, head) slice of the workload's recipe drawn on the host
    (numpy, rounded to bf16), for the reference arm, which has no GPU inputs:
    (q1, k1, q2, k2, g) as fp64 arrays."""
    import numpy as np
    rng = np.random.default_rng(seed)

    def bf16(x):
        # round fp32 draws to bf16 (nearest-even on the bit pattern)
        u = x.astype(np.float32).view(np.uint32)
        u = ((u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
        return u.view(np.float32).astype(np.float64)

    q1 = bf16(rng.standard_normal((w.NQ, w.d)) * w.teacher_std)
    k1 = bf16(rng.standard_normal((w.NK, w.d)) * w.teacher_std)
    q2 = bf16(q1 + w.noise * rng.standard_normal((w.NQ, w.d)))
    k2 = bf16(k1 + w.noise * rng.standard_normal((w.NK, w.d)))
    g = np.full(w.NQ, 1.0 / (w.B * w.H * w.NQ))
    return q1, k1, q2, k2, g


def oracle_rows(w, head, rows):
    """The fp64 oracle (forward + backward with the workload's gradient sets)
    on query rows `rows` of one head given as host arrays. Returns
    (seconds, visible pairs, (kl, lse1, lse2), (dq2, dk2, dq1, dk1))."""
    import numpy as np
    from oracle import streamkl_oracle as orc
    q1, k1, q2, k2, g = head
    t0 = time.perf_counter()
    fwd = orc.head_forward(q1, k1, q2, k2, w.scale, w.causal, rows=rows)
    bwd = orc.head_backward(q1, k1, q2, k2, w.scale, w.causal, g, w.grad1, rows=rows)
    dt = time.perf_counter() - t0
    off = w.NK - w.NQ
    pairs = int(np.sum(np.minimum(w.NK, rows + 1 + off))) if w.causal else len(rows) * w.NK
    return dt, pairs, fwd, bwd


def oracle_sample(w, budget_s: float, head):
    """Time the oracle on the last R query rows of one head, doubling R until
    the sample takes about budget_s / 3 seconds. Returns (TFLOP/s in the
    metric's convention on the sample's visible pairs, seconds, rows, oracle
    outputs, description)."""
    import numpy as np
    r = 64
    while True:
        rows = np.arange(w.NQ - r, w.NQ)
        dt, pairs, fwd, bwd = oracle_rows(w, head, rows)
        # metric convention on the exact pairs of the sample: (4 + 8) d per pair
        flops = 12.0 * pairs * w.d
        if dt >= budget_s / 3 or r >= w.NQ:
            desc = (f"last {r} query rows of one head (all their {pairs} visible (query,key) "
                    f"pairs), forward + backward"
                    f"{' with both gradient sets' if w.grad1 else ''}, fp64 numpy")
            return flops / dt / 1e12, dt, rows, (fwd, bwd), desc
        r = min(w.NQ, r * 2)


def cpu_cores():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:  # noqa: BLE001
        pass
    return os.cpu_count() or 1


def _rel_l2(got, ref):
    import numpy as np
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def error_stats(w, rows, oracle_out, gpu_head):
    """The GPU results of one head against the oracle's on `rows`: KL as the
    largest |error| / (2e-3 + 1e-2 |ref|) (pass <= 1), relative L2 of LSE1,
    LSE2 and of each gradient (pass <= 1e-4 and 1e-2). dK is compared on the
    keys that only `rows` see (all keys when rows are all rows; the last
    len(rows) keys under the causal mask), where a row sample gives it
    exactly."""
    import numpy as np
    (okl, ol1, ol2), og = oracle_out
    kl, l1, l2, grads = gpu_head
    err = np.abs(kl[rows] - okl)
    st = {"kl_max_err_over_bound": float(np.max(err / (2e-3 + 1e-2 * np.abs(okl)))),
          "lse1_rel_l2": _rel_l2(l1[rows], ol1), "lse2_rel_l2": _rel_l2(l2[rows], ol2)}
    if len(rows) == w.NQ:
        keys = np.arange(w.NK)
    elif w.causal:
        keys = np.arange(w.NK - len(rows), w.NK)
    else:
        keys = None
    names = ["dq2", "dk2", "dq1", "dk1"]
    for i, name in enumerate(names):
        if grads[i] is None or og[i] is None:
            continue
        if name.startswith("dq"):
            st[f"{name}_rel_l2"] = _rel_l2(grads[i][rows], og[i])
        elif keys is not None:
            st[f"{name}_rel_l2"] = _rel_l2(grads[i][keys], og[i][keys])
    st["dk_keys_compared"] = 0 if keys is None else int(len(keys))
    st["pass"] = bool(st["kl_max_err_over_bound"] <= 1.0 and st["lse1_rel_l2"] <= 1e-4
                      and st["lse2_rel_l2"] <= 1e-4
                      and all(v <= 1e-2 for k, v in st.items() if k.startswith("d")
                              and k.endswith("_rel_l2")))
    return st


def host_head(tensors, b, h):
    """fp64 host copies of slice (b, h) of device tensors (None stays None)."""
    return [None if t is None else t[b, h].float().cpu().numpy().astype("float64")
            for t in tensors]


# --------------------------------------------------------------------------- arms
def emit(obj):
    print(json.dumps(obj), flush=True)


def reference_arm(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    budget = args.cpu_budget_s
    head = draw_head(w)
    for _ in range(args.warmup):
        oracle_sample(w, min(budget, 2.0), head)
    vals, times = [], []
    desc = ""
    for _ in range(args.steps):
        v, dt, _, _, desc = oracle_sample(w, budget / max(1, args.steps), head)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    emit({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"head 0 of a host draw of the recipe, {desc}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    })
    return 0


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu capture
    (profiles/dram_traffic.json), or None when there is none for this workload
    or the kernel's sources have changed since it was taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return None
    for e in doc.get("entries", []):
        if e.get("workload") != workload or e.get("kernel") != kernel:
            continue
        h = hashlib.sha256()
        try:
            for src in e["sources"]:
                with open(os.path.join(ROOT, src), "rb") as f:
                    h.update(f.read())
        except OSError:
            return None
        return float(e["bytes_per_launch"]) if h.hexdigest() == e.get("sha256") else None
    return None


def describe(w):
    return (f"{w.name}: B={w.B} H={w.H} N_Q={w.NQ} N_K={w.NK} d={w.d} "
            f"{'causal' if w.causal else 'non-causal'}, bf16 inputs, fwd+bwd"
            f"{' incl. dQ1,dK1' if w.grad1 else ''}")


def _time_calls(fn, reps, stream):
    import torch
    fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return statistics.median(out)


# Oracle sample per named workload in the per-config entries: which head and
# how many of its last query rows (None: all rows; all heads for "tiny").
CONFIG_SAMPLES = {"tiny": None, "mid": ((1, 15), None), "splitk": ((3, 31), None),
                  "stress": ((0, 7), 1024)}


def config_entry(w, binding, synthetic, dev, pk, seed):
    """One named workload at full size: forward and backward times (median of
    3 timed calls after one untimed, CUDA events, inputs resident), method
    and executed TFLOP/s, and the error against the oracle on a sample."""
    import numpy as np
    import torch
    q1, k1, q2, k2, g = synthetic.make_inputs(w, seed, dev)
    B, H, NQ, NK, d = w.B, w.H, w.NQ, w.NK, w.d
    ws_bytes = binding.streamkl_workspace_size(B, H, NQ, NK, d, w.causal, w.grad1)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    status = binding.new_status(dev)
    outs = tuple(torch.empty((B, H, NQ), dtype=torch.float32, device=dev) for _ in range(3))
    grads = (torch.empty_like(q2), torch.empty_like(k2),
             torch.empty_like(q1) if w.grad1 else None, torch.empty_like(k1) if w.grad1 else None)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, out=outs, workspace=ws,
                             dev_status=status)

    def bwd():
        binding.streamkl_bwd(q1, k1, q2, k2, *outs, g, w.scale, w.causal, grad1=w.grad1, out=grads,
                             workspace=ws, dev_status=status)

    fwd_ms = _time_calls(fwd, 3, stream)
    bwd_ms = _time_calls(bwd, 3, stream)
    binding.raise_on_device_status(status, w.name)
    separate = binding.bwd_algorithm(B, H, NQ, NK, d, w.causal, w.grad1) == binding.BWD_SEPARATE
    mf, mb = method_flops(w)
    xb = executed_bwd_flops(w, separate)
    sus = pk["bf16_tflops_sustained"]
    e = {"workload": describe(w), "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
         "fwd_tflops": mf / fwd_ms / 1e9, "bwd_tflops_method": mb / bwd_ms / 1e9,
         "bwd_tflops_executed": xb / bwd_ms / 1e9,
         "frac_of_measured_sustained": {"fwd": mf / fwd_ms / 1e9 / sus,
                                        "bwd_method": mb / bwd_ms / 1e9 / sus}}
    # the oracle on a sample of the same inputs (the CPU-baseline leg's work)
    plan = CONFIG_SAMPLES.get(w.name)
    heads = [(b, h) for b in range(B) for h in range(H)] if plan is None else [plan[0]]
    r = None if plan is None else plan[1]
    stats, secs = [], 0.0
    for (b, h) in heads:
        head = host_head((q1, k1, q2, k2, g), b, h)
        rows = np.arange(NQ) if r is None else np.arange(NQ - r, NQ)
        dt, _, fo, bo = oracle_rows(w, head, rows)
        secs += dt
        gpu = host_head(outs + grads, b, h)
        stats.append(error_stats(w, rows, (fo, bo), (gpu[0], gpu[1], gpu[2], gpu[3:])))
    worst = {k: max(s[k] for s in stats) for k in stats[0] if k not in ("pass",)}
    worst["pass"] = all(s["pass"] for s in stats)
    e["oracle"] = {"sample": (f"heads {heads}, " + ("all query rows" if r is None
                                                     else f"last {r} query rows")),
                   "seconds": secs, "errors": worst}
    del q1, k1, q2, k2, g, ws, outs, grads
    torch.cuda.empty_cache()
    return e


def gpu_arm(args, w):
    import torch
    from attention_kl_loss_gb300 import binding, synthetic

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist_init("nccl")
    binding.load()
    q1, k1, q2, k2, g = synthetic.make_inputs(w, replica_seed(rank), dev)
    B, H, NQ, NK, d = w.B, w.H, w.NQ, w.NK, w.d
    ws_bytes = binding.streamkl_workspace_size(B, H, NQ, NK, d, w.causal, w.grad1)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    status = binding.new_status(dev)
    kl, l1, l2 = (torch.empty((B, H, NQ), dtype=torch.float32, device=dev) for _ in range(3))
    grads = (torch.empty_like(q2), torch.empty_like(k2),
             torch.empty_like(q1) if w.grad1 else None, torch.empty_like(k1) if w.grad1 else None)
    splits = binding.choose_splits(B, H, NQ, NK, d, w.causal)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, out=(kl, l1, l2), workspace=ws,
                             dev_status=status)
        if ev is not None:
            ev[1].record(stream)
        binding.streamkl_bwd(q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal, grad1=w.grad1,
                             out=grads, workspace=ws, dev_status=status)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    binding.raise_on_device_status(status, "warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize(dev)
        start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        stop.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
    binding.raise_on_device_status(status, "timed region")
    clocks = clk.summary()
    ms_total = start.elapsed_time(stop)
    ms_total = max_over_ranks(ms_total, dev)
    ms_step = ms_total / args.steps
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)

    f_fwd, f_bwd_metric = flop_counts(w)
    m_fwd, m_bwd = method_flops(w)
    algo = binding.bwd_algorithm(B, H, NQ, NK, d, w.causal, w.grad1)
    separate = algo == binding.BWD_SEPARATE
    x_bwd = executed_bwd_flops(w, separate)
    pairs = w.live_pairs_per_head() * B * H
    if separate:
        bwd_name = "streamkl_bwd_sep_kernel (dK + dQ)"
        bwd_note = ("separate dK and dQ kernels, timed together (one API call); each "
                    "regenerates S1 and S2, so they execute 16d FLOPs per pair with both "
                    "gradient sets against the method's 12d")
    elif NQ <= 64 and d == 128:
        bwd_name = "streamkl_bwd_short_kernel"
        bwd_note = ("fused algorithm, short-sweep kernel (each pair visited once, dQ kept on chip "
                    "per batch-head); includes the workspace clear and the fp32->bf16 dQ "
                    "conversion; bound by HBM")
    else:
        bwd_name = "streamkl_bwd_fused_kernel" if d == 64 else "streamkl_bwd_fused128_kernel"
        bwd_note = ("fused algorithm, one CTA per key tile (each pair visited once, dQ added with "
                    "TMA bulk reductions); includes the workspace clear and the fp32->bf16 dQ "
                    "conversion")
    short_sweep = (not separate) and NQ <= 64 and d == 128
    step_flops = f_fwd + f_bwd_metric
    value = world * step_flops / (ms_step * 1e-3) / 1e12
    pk = peaks()
    sustained, burst = pk["bf16_tflops_sustained"], pk["bf16_tflops"]
    fwd_tf = m_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = m_bwd / (bwd_ms * 1e-3) / 1e12
    bwd_xtf = x_bwd / (bwd_ms * 1e-3) / 1e12
    unit_note = ("method work on the exact visible (query, key) pairs: forward 4d FLOPs per "
                 "pair; backward 4d (regenerate S1, S2) + 4d per gradient set")
    kernels = {
        "streamkl_fwd_kernel": {"ms": fwd_ms, "algorithmic_tflop": m_fwd / 1e12,
                                "achieved_tflops": fwd_tf,
                                "frac_of_measured_sustained": fwd_tf / sustained,
                                "frac_of_measured_burst": fwd_tf / burst},
        bwd_name: {"ms": bwd_ms, "algorithmic_tflop": m_bwd / 1e12,
                   "achieved_tflops": bwd_tf, "frac_of_measured_sustained": bwd_tf / sustained,
                   "frac_of_measured_burst": bwd_tf / burst,
                   "executed_tflop": x_bwd / 1e12, "executed_tflops": bwd_xtf,
                   "executed_frac_of_measured_sustained": bwd_xtf / sustained,
                   "note": bwd_note},
    }
    dom = bwd_name if bwd_ms >= fwd_ms else "streamkl_fwd_kernel"
    dom_tf = kernels[dom]["achieved_tflops"]
    traffic = recorded_traffic(w.name, dom)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": dom_tf, "peak": sustained,
                "unit": "TFLOP/s", "frac": dom_tf / sustained, "traffic": traffic,
                "algorithmic": unit_note,
                "peak_source": f"{pk['source']} bf16_tflops_sustained (kernel timed inside a long step)",
                "frac_of_measured_burst": dom_tf / burst}
    if dom == bwd_name and short_sweep:
        # the short-sweep backward moves the keys once and writes dK: HBM-bound
        mb = bwd_min_bytes(w)
        gbs = mb / (bwd_ms * 1e-3) / 1e9
        roofline.update({"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / pk["hbm_gbs"],
                         "algorithmic": "minimum bytes of the backward: Q1, K1, Q2, K2 read once, "
                                        "the gradients written once, the per-row vectors read",
                         "peak_source": f"{pk['source']} hbm_gbs (copy bandwidth)",
                         "tensor_tflops": bwd_tf})
        roofline.pop("frac_of_measured_burst", None)
    elif dom == bwd_name:
        roofline["executed_tflops"] = bwd_xtf
        roofline["executed_frac"] = bwd_xtf / sustained
        if traffic is not None:
            mb = bwd_min_bytes(w)
            roofline["traffic_min_bytes"] = mb
            roofline["traffic_over_min"] = traffic / mb
            roofline["traffic_ok"] = traffic <= 1.5 * mb
            if traffic > 1.5 * mb:
                print(f"warning: {dom} moves {traffic / mb:.2f}x its minimum DRAM bytes "
                      "(limit 1.5x)", file=sys.stderr)
    if separate:
        launches_per_step = 1 + (1 if splits > 1 else 0) + 2
    else:
        launches_per_step = 1 + (1 if splits > 1 else 0) + 1 + (2 if w.grad1 else 1)

    e2e = None
    if not args.no_e2e:
        e2e = e2e_measure(args, w, binding, synthetic, dev, rank, step_flops, world)

    cpu = None
    configs = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        head = host_head((q1, k1, q2, k2, g), 0, 0)
        v, dt, rows, oo, desc = oracle_sample(w, args.cpu_budget_s, head)
        gpu = host_head((kl, l1, l2) + grads, 0, 0)
        main_err = error_stats(w, rows, oo, (gpu[0], gpu[1], gpu[2], gpu[3:]))
        cpu = {"value": v, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"head 0 of the timed run's inputs, {desc}; {dt:.1f} s"}
        configs = [{"workload": describe(w), "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
                    "fwd_tflops": fwd_tf, "bwd_tflops_method": bwd_tf,
                    "bwd_tflops_executed": bwd_xtf,
                    "frac_of_measured_sustained": {"fwd": fwd_tf / sustained,
                                                   "bwd_method": bwd_tf / sustained},
                    "oracle": {"sample": f"head 0, last {len(rows)} query rows", "seconds": dt,
                               "errors": main_err}}]
        if not args.no_configs:
            del q1, k1, q2, k2, g, ws, grads
            torch.cuda.empty_cache()
            for i, name in enumerate(("tiny", "mid", "splitk", "stress")):
                if name != w.name:
                    configs.append(config_entry(synthetic.WORKLOADS[name], binding, synthetic,
                                                dev, pk, 2000 + i))

    extra_hbm = {
        "workspace_bytes": ws_bytes,
        "saved_state_bytes": 3 * B * H * NQ * 4,
        "materialised_p1_p2_bytes_avoided": 2 * B * H * NQ * NK * 2,
    }
    if rank == 0:
        emit({
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": describe(w), "B": B, "H": H, "N_Q": NQ, "N_K": NK, "d": d,
                       "causal": w.causal, "grad1": w.grad1, "splits": splits,
                       "bwd_algorithm": "separate" if separate else "fused",
                       "flop_convention": "4 NQ NK d fwd + 8 NQ NK d bwd per head, halved for causal",
                       "l2": l2_note(B, H, NQ, NK, d), "parallelism": f"replicas x{world}"},
            "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
            "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
            "bwd_tflops_metric": f_bwd_metric / (bwd_ms * 1e-3) / 1e12,
            # the same times over the method's work on the exact visible pairs
            "visible_pairs": pairs,
            "fwd_tflops_method": fwd_tf,
            "bwd_tflops_method": bwd_tf,
            "pct_of_measured_peak": {"value": value / world / burst,
                                     "fwd": f_fwd / (fwd_ms * 1e-3) / 1e12 / burst,
                                     "bwd_metric": f_bwd_metric / (bwd_ms * 1e-3) / 1e12 / burst,
                                     "peak": f"{pk['source']} bf16_tflops (burst)"},
            "roofline": roofline, "kernels": kernels,
            "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "gpu_launches": launches_per_step * args.steps,
            "extra_hbm": extra_hbm,
            "configs": configs,
        })
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def e2e_measure(args, w, binding, synthetic, dev, rank, step_flops, world):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and every result back to pinned host
    memory (KL, LSE1, LSE2 and the gradients).

    A step's batch goes through the API in G groups of (batch, head) slices
    (heads are independent, so this is the same computation), streamed
    through two device slots: group u's inputs are copied in on one stream
    and its results out on another, so group u+1's inputs and group u-1's
    results move while group u computes. Every copy is enqueued after the
    start event and the stop event waits for the last one, so all of them
    fall inside the timed region."""
    import torch
    q1, k1, q2, k2, g = synthetic.make_inputs(w, replica_seed(rank) + 7, dev)
    host_in = [t.cpu().pin_memory() for t in (q1, k1, q2, k2, g)]
    del q1, k1, q2, k2, g
    bh = w.B * w.H
    groups = next(c for c in (args.e2e_groups, 4, 2, 1) if c >= 1 and bh % c == 0)
    per = bh // groups

    def part(t, i):  # slices [i per, (i+1) per) of the flattened (batch, head) axis, as [1, per, ...]
        return t.reshape((bh,) + tuple(t.shape[2:]))[i * per:(i + 1) * per].unsqueeze(0)

    host_groups = [[part(t, i) for t in host_in] for i in range(groups)]
    # results on the host: kl, lse1, lse2, then dq2, dk2 (and dq1, dk1)
    row = torch.empty((w.B, w.H, w.NQ), dtype=torch.float32)
    host_out = [torch.empty_like(row).pin_memory() for _ in range(3)]
    host_out += [torch.empty_like(host_in[2]).pin_memory(), torch.empty_like(host_in[3]).pin_memory()]
    if w.grad1:
        host_out += [torch.empty_like(host_in[0]).pin_memory(),
                     torch.empty_like(host_in[1]).pin_memory()]
    host_out_groups = [[part(t, i) for t in host_out] for i in range(groups)]
    in_bufs = [[torch.empty_like(t, device=dev) for t in host_groups[0]] for _ in range(2)]
    out_bufs = [[torch.empty_like(t, device=dev) for t in host_out_groups[0]] for _ in range(2)]
    sub = host_groups[0]
    ws_bytes = binding.streamkl_workspace_size(1, per, w.NQ, w.NK, w.d, w.causal, w.grad1)
    ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
    status = binding.new_status(dev)
    stream = torch.cuda.current_stream(dev)
    h2d_stream = torch.cuda.Stream(dev)
    d2h_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(2)]     # inputs of a slot copied in
    in_free = [torch.cuda.Event() for _ in range(2)]   # a slot's inputs consumed
    done = [torch.cuda.Event() for _ in range(2)]      # a slot's results computed
    out_free = [torch.cuda.Event() for _ in range(2)]  # a slot's results copied out
    assert sub[0].shape[1] == per

    def h2d(slot, gi):
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(in_free[slot])
            for hsrc, d in zip(host_groups[gi], in_bufs[slot]):
                d.copy_(hsrc, non_blocking=True)
            ready[slot].record(h2d_stream)

    def d2h(slot, gi):
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(done[slot])
            for d, hdst in zip(out_bufs[slot], host_out_groups[gi]):
                hdst.copy_(d, non_blocking=True)
            out_free[slot].record(d2h_stream)

    def run(steps):
        for e in in_free + out_free:
            e.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        units = steps * groups
        h2d(0, 0)
        for u in range(units):
            slot, gi = u & 1, u % groups
            if u + 1 < units:
                h2d(slot ^ 1, (u + 1) % groups)
            stream.wait_event(ready[slot])
            stream.wait_event(out_free[slot])
            x, o = in_bufs[slot], out_bufs[slot]
            binding.streamkl_fwd(*x[:4], w.scale, w.causal, out=tuple(o[:3]), workspace=ws,
                                 dev_status=status)
            binding.streamkl_bwd(*x[:4], *o[:3], x[4], w.scale, w.causal, grad1=w.grad1,
                                 out=tuple(o[3:]) + ((None, None) if not w.grad1 else ()),
                                 workspace=ws, dev_status=status)
            in_free[slot].record(stream)
            done[slot].record(stream)
            d2h(slot, gi)
        stream.wait_stream(d2h_stream)

    run(max(1, args.warmup))
    torch.cuda.synchronize(dev)
    binding.raise_on_device_status(status, "e2e warm-up")
    barrier()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(args.steps)
    b.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    binding.raise_on_device_status(status, "e2e")
    ms = max_over_ranks(a.elapsed_time(b) / args.steps, dev)
    h2d_bytes = sum(t.numel() * t.element_size() for t in host_in)
    d2h_bytes = sum(t.numel() * t.element_size() for t in host_out)
    return {"value": world * step_flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
            "results_copied": "kl, lse1, lse2, dq2, dk2" + (", dq1, dk1" if w.grad1 else ""),
            "overlap": f"each step's batch in {groups} groups of {per} (batch, head) slices through "
                       "two device slots: a group's inputs are copied in on one stream and its "
                       "results out on another while the neighbouring group computes",
            "api": "attention_kl_loss_gb300.streamkl_fwd/streamkl_bwd (ctypes over the C ABI)"}


def l2_note(B, H, NQ, NK, d):
    """How the timed steps relate to the 129 MB L2: the four bf16 inputs'
    size (no flush runs between steps)."""
    in_bytes = 2 * 2 * B * H * (NQ + NK) * d
    rel = "larger" if in_bytes > 129e6 else "not larger"
    return f"inputs ({in_bytes / 1e6:.0f} MB) {rel} than the 129 MB L2; no flush"


def main(argv=None):
    args = parse_args(argv)
    from attention_kl_loss_gb300 import synthetic
    w = synthetic.WORKLOADS[args.workload]
    if args.impl == "reference":
        return reference_arm(args, w)
    if args.warmup < 3:
        print("note: fewer than 3 warm-up steps requested", file=sys.stderr)
    return gpu_arm(args, w)


if __name__ == "__main__":
    sys.exit(main())
