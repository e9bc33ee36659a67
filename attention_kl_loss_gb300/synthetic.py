"""Seeded synthetic inputs for the attention-KL primitive.

This module only draws random tensors; it holds none of the method's
arithmetic. Both the CUDA path and the fp64 oracle are fed from it (the oracle
receives a host copy of exactly the bf16 values the GPU sees).

The named workloads stand in for the context-length sweeps of the pages'
evaluation ("Resultados Experimentales": 4K to 512K contexts; the problem
statement's 64K-context, 32-head BF16 example). Recipe, per workload:

* teacher Q1, K1 ~ teacher_std * N(0, 1), drawn in fp32;
* student either teacher + noise * N(0, 1) (added to the fp32 draw) or an
  independent student_std * N(0, 1) draw;
* all four rounded to bf16 (round-to-nearest-even) and laid out [B, H, N, d];
* upstream per-row gradient g = 1 / (B * H * N_Q) (a mean over rows);
* scale = 1 / sqrt(d).

Draws use ``torch.Generator`` on the requested device, seeded per call, in a
fixed order (Q1, K1, then the student draws), so a seed names one input set
per device type.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    NQ: int
    NK: int
    d: int
    causal: bool
    teacher_std: float = 1.0
    student: str = "noise"  # "noise": teacher + noise*eps; "independent": student_std*eps
    noise: float = 0.1
    student_std: float = 1.0
    grad1: bool = False  # also produce dQ1, dK1 (configuration 2 gradients)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def live_pairs_per_head(self) -> int:
        """Exact count of unmasked (query, key) pairs in one (b, h) slice."""
        if not self.causal:
            return self.NQ * self.NK
        off = self.NK - self.NQ
        # row i sees i + 1 + off keys (never more than NK since off = NK - NQ)
        return self.NQ * (self.NQ + 1) // 2 + self.NQ * off


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", B=1, H=2, NQ=256, NK=256, d=64, causal=False, noise=0.3),
        Workload("mid", B=2, H=16, NQ=4096, NK=4096, d=128, causal=False, noise=0.1),
        Workload("causal64k", B=1, H=32, NQ=65536, NK=65536, d=128, causal=True,
                 noise=0.2, grad1=True),
        Workload("splitk", B=4, H=32, NQ=512, NK=131072, d=128, causal=True, noise=0.1),
        Workload("stress", B=1, H=8, NQ=16384, NK=16384, d=64, causal=False,
                 teacher_std=3.0, student="independent", student_std=1.0),
        # smaller causal case with the 64K workload's tile mix, sized for
        # profiler captures (256 MiB of inputs: above L2, a few GB at most)
        Workload("causal16k_profile", B=1, H=16, NQ=16384, NK=16384, d=128, causal=True,
                 noise=0.2, grad1=True),
        # the 64K causal shape on 4 heads: DRAM-traffic captures, whose per-head
        # traffic and work are those of the full 32-head workload
        Workload("causal64k_h4", B=1, H=4, NQ=65536, NK=65536, d=128, causal=True, noise=0.2,
                 grad1=True),
        # the split-K shape on 4 of its 32 heads (keys 1.07 GB, above L2):
        # DRAM-traffic captures of the split forward
        Workload("splitk_h4", B=4, H=4, NQ=512, NK=131072, d=128, causal=True, noise=0.1),
        # a decode-like shape (64 query rows against 64K keys) on 8 heads, for
        # profiler captures of the fused short-sweep backward (keys 268 MB)
        Workload("decode_profile", B=1, H=8, NQ=64, NK=65536, d=128, causal=True, noise=0.1),
        # d = 64, one gradient set, causal 16K on 16 heads (inputs 134 MB, above
        # L2): profiler captures of the fused d = 64 backward
        Workload("causal16k_d64_profile", B=1, H=16, NQ=16384, NK=16384, d=64, causal=True,
                 noise=0.2),
    ]
}


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit sizes (used for ragged and edge-case tests)."""
    return Workload(name=name, **kw)


def make_inputs(w: Workload, seed: int = 0, device="cpu"):
    """Return (q1, k1, q2, k2, g): bf16 [B,H,N,d] x4 and fp32 g [B,H,N_Q]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    sq = (w.B, w.H, w.NQ, w.d)
    sk = (w.B, w.H, w.NK, w.d)

    def draw(shape):
        return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)

    q1f = draw(sq).mul_(w.teacher_std)
    k1f = draw(sk).mul_(w.teacher_std)
    if w.student == "noise":
        q2f = draw(sq).mul_(w.noise).add_(q1f)
        k2f = draw(sk).mul_(w.noise).add_(k1f)
    elif w.student == "independent":
        q2f = draw(sq).mul_(w.student_std)
        k2f = draw(sk).mul_(w.student_std)
    else:
        raise ValueError(f"unknown student mode {w.student!r}")
    q1, k1, q2, k2 = (t.to(torch.bfloat16) for t in (q1f, k1f, q2f, k2f))
    del q1f, k1f, q2f, k2f
    g = torch.full((w.B, w.H, w.NQ), 1.0 / (w.B * w.H * w.NQ), device=device,
                   dtype=torch.float32)
    return q1, k1, q2, k2, g


def make_packed_inputs(lens_q, lens_k, H: int, d: int, seed: int = 0, noise: float = 0.3,
                       device="cpu"):
    """A packed variable-length batch: sequence b has lens_q[b] query rows and
    lens_k[b] key rows. Returns (q1, k1, q2, k2, g, cu_q, cu_k): bf16
    [total, H, d] x4 (teacher ~ N(0,1), student = teacher + noise N(0,1)),
    fp32 g [total_q, H] = 1 / (H total_q), int32 offsets [B + 1]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    tq, tk = int(sum(lens_q)), int(sum(lens_k))

    def draw(rows):
        return torch.randn((rows, H, d), generator=gen, device=device, dtype=torch.float32)

    q1f, k1f = draw(tq), draw(tk)
    q2f = draw(tq).mul_(noise).add_(q1f)
    k2f = draw(tk).mul_(noise).add_(k1f)
    q1, k1, q2, k2 = (t.to(torch.bfloat16) for t in (q1f, k1f, q2f, k2f))
    g = torch.full((tq, H), 1.0 / (H * max(tq, 1)), device=device, dtype=torch.float32)

    def offsets(lens):
        cu = [0]
        for n in lens:
            cu.append(cu[-1] + int(n))
        return torch.tensor(cu, dtype=torch.int32, device=device)

    return q1, k1, q2, k2, g, offsets(lens_q), offsets(lens_k)
