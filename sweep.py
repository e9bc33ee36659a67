"""Sweeps behind the design choices (run on one GPU, prints markdown tables).

    python sweep.py algo      # fused vs separate backward
    python sweep.py decode    # split-K on/off for few query rows
    python sweep.py context   # context length 4K .. 512K
    python sweep.py dqsplit   # backward dQ key split on/off
    python sweep.py configs   # the named workloads, fwd and bwd
    python sweep.py dkpersist # persistent dK kernel off/on, short queries

Every point is timed through the C ABI with CUDA events on the current stream,
inputs resident in device memory, one untimed call first, the median of
``--reps`` timed calls reported. Inputs are the synthetic recipe of
``synthetic.make_inputs`` (teacher ~ N(0,1), student = teacher + noise).
FLOP counts use the exact number of visible (query, key) pairs: 4d per pair
forward; backward 8d per pair and gradient set (two score recomputes, dK, dQ).
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_kl_loss_gb300 import binding, synthetic  # noqa: E402


def _time(fn, reps: int) -> float:
    fn()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        out.append(a.elapsed_time(b))
    return statistics.median(out)


def _setup(w, dev):
    q1, k1, q2, k2, g = synthetic.make_inputs(w, 0, dev)
    status = binding.new_status(dev)
    return (q1, k1, q2, k2, g), status


def _check(status, where):
    binding.raise_on_device_status(status, where)


def sweep_algo(reps: int):
    """The fused algorithm (at most 64 query rows at d = 128: the short-sweep
    kernel with dQ kept on chip per batch-head; at d = 64 one CTA per key tile
    with dQ through TMA reductions; otherwise one CTA per key tile with dQ
    through fp32 L2 reductions) against the separate dK/dQ kernels."""
    dev = torch.device("cuda")
    shapes = [synthetic.WORKLOADS[n] for n in ("mid", "stress", "splitk", "causal64k")] + [
        synthetic.custom("decode64", B=4, H=32, NQ=64, NK=65536, d=128, causal=True, noise=0.1),
        synthetic.custom("decode64_both", B=4, H=32, NQ=64, NK=65536, d=128, causal=True,
                         noise=0.1, grad1=True),
        synthetic.custom("decode1", B=4, H=32, NQ=1, NK=65536, d=128, causal=True, noise=0.1),
        synthetic.custom("decode16_128k", B=4, H=32, NQ=16, NK=131072, d=128, causal=True,
                         noise=0.1),
        synthetic.custom("decode32_nc", B=1, H=32, NQ=32, NK=32768, d=128, causal=False,
                         noise=0.1),
        synthetic.custom("square16k_d64", B=1, H=16, NQ=16384, NK=16384, d=64, causal=True,
                         noise=0.2, grad1=True),
        synthetic.custom("square8k", B=2, H=16, NQ=8192, NK=8192, d=128, causal=False, noise=0.2,
                         grad1=True),
    ] + [synthetic.custom(f"short{nq}x{nk // 1024}k", B=4, H=32, NQ=nq, NK=nk, d=128, causal=True,
                          noise=0.1)
         for nq in (256, 1024, 2048) for nk in (65536, 131072)] + [
        # d = 64, one gradient set: the fused kernel with dQ through TMA reductions
        synthetic.custom(f"d64_{nq}x{nk // 1024}k", B=b, H=h, NQ=nq, NK=nk, d=64, causal=causal,
                         noise=0.2)
        for (b, h, nq, nk, causal) in [(4, 32, 64, 65536, True), (4, 32, 128, 65536, True),
                                       (4, 32, 256, 65536, True), (1, 8, 512, 131072, True),
                                       (2, 16, 1024, 1024, False), (2, 16, 2048, 2048, True),
                                       (2, 16, 4096, 4096, False), (1, 16, 16384, 16384, True),
                                       (1, 8, 65536, 65536, True)]] + [
        # d = 128, moderate key lengths: the fused kernel's dQ reductions against
        # the separate kernels' second pass over the scores
        synthetic.custom(f"d128_{nq}x{nk // 1024}k", B=b, H=h, NQ=nq, NK=nk, d=128, causal=causal,
                         noise=0.2, grad1=g1)
        for (b, h, nq, nk, causal, g1) in [(2, 16, 2048, 2048, False, False),
                                           (4, 32, 2048, 2048, True, False),
                                           (2, 16, 8192, 8192, False, False),
                                           (1, 16, 16384, 16384, True, False),
                                           (2, 16, 4096, 4096, False, True),
                                           (4, 16, 2048, 8192, True, False),
                                           (4, 32, 256, 8192, False, False),
                                           (4, 32, 512, 2048, False, False),
                                           (4, 32, 512, 16384, False, False),
                                           (2, 16, 1024, 32768, False, False),
                                           (1, 16, 16384, 16384, False, False)]]
    print("| workload | sets | separate ms | fused ms | faster | library's choice |")
    print("|---|---|---:|---:|---|---|")
    for w in shapes:
        (q1, k1, q2, k2, g), st = _setup(w, dev)
        kl, l1, l2 = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, dev_status=st)
        res = {}
        for algo in (binding.BWD_SEPARATE, binding.BWD_FUSED):
            binding.set_bwd_algorithm(algo)
            try:
                res[algo] = _time(lambda: binding.streamkl_bwd(
                    q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal, grad1=w.grad1,
                    dev_status=st), reps)
            finally:
                binding.set_bwd_algorithm(None)
        _check(st, w.name)
        choice = binding.bwd_algorithm(w.B, w.H, w.NQ, w.NK, w.d, w.causal, w.grad1)
        sep, fus = res[binding.BWD_SEPARATE], res[binding.BWD_FUSED]
        print(f"| {w.name} (B{w.B} H{w.H} {w.NQ}x{w.NK} d{w.d}{' causal' if w.causal else ''}) "
              f"| {'both' if w.grad1 else 'config 1'} | {sep:.3f} | {fus:.3f} | "
              f"{'separate' if sep <= fus else 'fused'} | "
              f"{'separate' if choice == binding.BWD_SEPARATE else 'fused'} |")
        del q1, k1, q2, k2, g
        torch.cuda.empty_cache()


def sweep_decode(reps: int):
    """Forward with few query rows against a long key range: split-K off / chosen."""
    dev = torch.device("cuda")
    print("| N_Q | N_K | splits chosen | ms, no split | ms, chosen | speed-up |")
    print("|---:|---:|---:|---:|---:|---:|")
    for nq in (1, 16, 64, 256, 512, 1024):
        for nk in (65536, 131072):
            w = synthetic.custom(f"decode{nq}", B=4, H=32, NQ=nq, NK=nk, d=128, causal=True,
                                 noise=0.1)
            (q1, k1, q2, k2, g), st = _setup(w, dev)
            s = binding.choose_splits(w.B, w.H, nq, nk, w.d, w.causal)
            t1 = _time(lambda: binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal,
                                                    num_splits=1, dev_status=st), reps)
            ts = _time(lambda: binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal,
                                                    num_splits=s, dev_status=st), reps)
            _check(st, w.name)
            print(f"| {nq} | {nk} | {s} | {t1:.3f} | {ts:.3f} | {t1 / ts:.2f} |")
            del q1, k1, q2, k2, g
            torch.cuda.empty_cache()


def sweep_dqsplit(reps: int):
    """Separate backward with the dQ kernel's key split forced off and at the
    library's choice, on shapes with few query blocks against long keys."""
    dev = torch.device("cuda")
    shapes = [synthetic.WORKLOADS["splitk"], synthetic.WORKLOADS["splitk_h4"]] + [
        synthetic.custom(f"q{nq}_k{nk // 1024}k_b{b}h{h}", B=b, H=h, NQ=nq, NK=nk, d=d, causal=True,
                         noise=0.1, grad1=g1)
        for (b, h, nq, nk, d, g1) in [(1, 8, 512, 131072, 128, False), (1, 32, 1024, 65536, 128, True),
                                      (4, 32, 256, 65536, 128, False), (4, 32, 64, 65536, 128, False),
                                      (1, 8, 512, 131072, 64, False)]]
    print("| workload | sets | splits chosen | ms, no split | ms, chosen | speed-up |")
    print("|---|---|---:|---:|---:|---:|")
    for w in shapes:
        (q1, k1, q2, k2, g), st = _setup(w, dev)
        kl, l1, l2 = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, dev_status=st)
        res = {}
        for forced in (1, None):
            binding.set_bwd_dq_splits(forced)
            binding.set_bwd_algorithm(binding.BWD_SEPARATE)  # 64 rows would go to the fused kernel
            try:
                res[forced] = _time(lambda: binding.streamkl_bwd(
                    q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal, grad1=w.grad1,
                    dev_status=st), reps)
            finally:
                binding.set_bwd_dq_splits(None)
                binding.set_bwd_algorithm(None)
        _check(st, w.name)
        s = binding.bwd_dq_splits(w.B, w.H, w.NQ, w.NK, w.d, w.causal, w.grad1)
        print(f"| {w.name} (B{w.B} H{w.H} {w.NQ}x{w.NK} d{w.d} causal) | "
              f"{'both' if w.grad1 else 'config 1'} | {s} | {res[1]:.3f} | {res[None]:.3f} | "
              f"{res[1] / res[None]:.2f} |")
        del q1, k1, q2, k2, g
        torch.cuda.empty_cache()


def sweep_dkpersist(reps: int):
    """Separate backward with the persistent dK kernel off and at the
    library's choice, for short query sweeps against long keys."""
    dev = torch.device("cuda")
    shapes = [synthetic.custom(f"q{nq}_k64k_b4h32", B=4, H=32, NQ=nq, NK=65536, d=128, causal=True,
                               noise=0.1) for nq in (64, 128, 256, 384, 512, 1024)] + [
        synthetic.custom("q128_k128k_b1h32", B=1, H=32, NQ=128, NK=131072, d=128, causal=True,
                         noise=0.1, grad1=True),
        synthetic.WORKLOADS["splitk"]]
    print("| workload | sets | persistent CTAs chosen | ms, off | ms, chosen | speed-up |")
    print("|---|---|---:|---:|---:|---:|")
    for w in shapes:
        (q1, k1, q2, k2, g), st = _setup(w, dev)
        kl, l1, l2 = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, dev_status=st)
        res = {}
        for forced in (-1, None):
            binding.set_bwd_dk_persist(forced)
            binding.set_bwd_algorithm(binding.BWD_SEPARATE)  # 64 rows would go to the fused kernel
            try:
                res[forced] = _time(lambda: binding.streamkl_bwd(
                    q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal, grad1=w.grad1,
                    dev_status=st), reps)
            finally:
                binding.set_bwd_dk_persist(None)
                binding.set_bwd_algorithm(None)
        _check(st, w.name)
        c = binding.bwd_dk_persist(w.B, w.H, w.NQ, w.NK, w.d, w.causal)
        print(f"| {w.name} (B{w.B} H{w.H} {w.NQ}x{w.NK} d{w.d} causal) | "
              f"{'both' if w.grad1 else 'config 1'} | {c} | {res[-1]:.3f} | {res[None]:.3f} | "
              f"{res[-1] / res[None]:.2f} |")
        del q1, k1, q2, k2, g
        torch.cuda.empty_cache()


def sweep_configs(reps: int):
    """Forward and backward of every named workload at the library's choices,
    with the exact visible-pair FLOP counts of the method's work: 4d per pair
    forward; backward 4d to regenerate S1, S2 plus 4d per gradient set (8d
    with one set, 12d with both). The separate backward executes 4d more
    (each of its two kernels regenerates both score tiles)."""
    import json
    dev = torch.device("cuda")
    peak = None
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            peak = json.load(f).get("bf16_tflops_sustained")
    print("| workload | sets | bwd algorithm | fwd ms | bwd ms | fwd TFLOP/s | bwd TFLOP/s method "
          "(executed) | fwd / bwd method of "
          f"{'measured sustained peak' if peak else 'peak (not available)'} |")
    print("|---|---|---|---:|---:|---:|---:|---|")
    for name in ("tiny", "mid", "causal64k", "splitk", "stress"):
        w = synthetic.WORKLOADS[name]
        (q1, k1, q2, k2, g), st = _setup(w, dev)
        out = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, dev_status=st)
        tf = _time(lambda: binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, out=out,
                                                dev_status=st), reps)
        kl, l1, l2 = out
        tb = _time(lambda: binding.streamkl_bwd(q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal,
                                                grad1=w.grad1, dev_status=st), reps)
        _check(st, name)
        pairs = w.live_pairs_per_head() * w.B * w.H
        sep = binding.bwd_algorithm(w.B, w.H, w.NQ, w.NK, w.d, w.causal, w.grad1) == binding.BWD_SEPARATE
        ff = 4 * w.d * pairs / tf / 1e9
        fm = (12 if w.grad1 else 8) * w.d * pairs / tb / 1e9
        fx = fm + (4 * w.d * pairs / tb / 1e9 if sep else 0.0)
        frac = f"{ff / peak:.2f} / {fm / peak:.2f}" if peak else "-"
        print(f"| {name} (B{w.B} H{w.H} {w.NQ}x{w.NK} d{w.d}{' causal' if w.causal else ''}) | "
              f"{'both' if w.grad1 else 'config 1'} | {'separate' if sep else 'fused'} | {tf:.3f} | "
              f"{tb:.3f} | {ff:.0f} | {fm:.0f} ({fx:.0f}) | {frac} |")
        del q1, k1, q2, k2, g
        torch.cuda.empty_cache()


def sweep_context(reps: int):
    """Causal fwd + bwd (both sets) from 4K to 512K: time and extra device memory."""
    dev = torch.device("cuda")
    print("| N | heads | fwd ms | bwd ms | fwd TFLOP/s | bwd TFLOP/s | inputs MiB | "
          "extra MiB (workspace + saved KL/LSE) | P1+P2 materialised, MiB |")
    print("|---:|---:|---:|---:|---:|---:|---:|---:|---:|")
    for n, h in ((4096, 32), (16384, 32), (65536, 32), (131072, 8), (262144, 4), (524288, 2)):
        w = synthetic.custom(f"ctx{n}", B=1, H=h, NQ=n, NK=n, d=128, causal=True, noise=0.2,
                             grad1=True)
        (q1, k1, q2, k2, g), st = _setup(w, dev)
        ws_bytes = binding.streamkl_workspace_size(1, h, n, n, 128, True, True)
        ws = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=dev)
        out = tuple(torch.empty((1, h, n), device=dev) for _ in range(3))
        grads = tuple(torch.empty_like(t) for t in (q2, k2, q1, k1))
        tf = _time(lambda: binding.streamkl_fwd(q1, k1, q2, k2, w.scale, True, out=out,
                                                workspace=ws, dev_status=st), reps)
        kl, l1, l2 = out
        tb = _time(lambda: binding.streamkl_bwd(q1, k1, q2, k2, kl, l1, l2, g, w.scale, True,
                                                grad1=True, out=grads, workspace=ws,
                                                dev_status=st), reps)
        _check(st, w.name)
        pairs = w.live_pairs_per_head() * h
        inputs = 4 * h * n * 128 * 2
        extra = ws_bytes + 3 * h * n * 4
        mat = 2 * h * n * n * 2
        print(f"| {n} | {h} | {tf:.3f} | {tb:.3f} | {4 * 128 * pairs / tf / 1e9:.0f} | "
              f"{16 * 128 * pairs / tb / 1e9:.0f} | {inputs / 2**20:.0f} | {extra / 2**20:.2f} | "
              f"{mat / 2**20:.0f} |")
        del q1, k1, q2, k2, g, grads, ws, out
        torch.cuda.empty_cache()


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("what", choices=["algo", "decode", "context", "dqsplit", "configs", "dkpersist"])
    p.add_argument("--reps", type=int, default=3)
    a = p.parse_args(argv)
    binding.load()
    {"algo": sweep_algo, "decode": sweep_decode, "context": sweep_context,
     "dqsplit": sweep_dqsplit, "configs": sweep_configs, "dkpersist": sweep_dkpersist}[a.what](a.reps)


if __name__ == "__main__":
    main()
