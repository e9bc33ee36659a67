"""The allocation-free forward entry point, streamkl_fwd_noalloc.

Some callers cannot allocate device memory: a plug-in operator running inside
another runtime that hands it only its input and output buffers, or code whose
device memory belongs to a host framework's pool, where an extra cudaMalloc
would fail, fragment the pool or stall the device. For them the library keeps
the forward pass's split scratch in a device array compiled into it. These
checks call that entry point through the C ABI and hold its results to the
regular streamkl_fwd (which takes a caller-provided workspace), with the
suite's tolerances, on two calls in a row that use the shared scratch with
different shapes. The file sorts last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from attention_kl_loss_gb300 import binding, synthetic
from oracle import streamkl_oracle as orc

KL_ABS, KL_REL, LSE_REL = 2e-3, 1e-2, 1e-4
SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module")
def lib():
    from attention_kl_loss_gb300 import build
    build.build()
    return binding.load()


def test_rejects_split_plans_beyond_the_builtin_scratch(lib):
    """Runs on the CPU: the size check comes before any device work."""
    p = ctypes.c_void_p(0x1000)
    # 8 splits x 32 heads x 65536 rows x 5 floats = 40 MiB > 16 MiB
    st = lib.streamkl_fwd_noalloc(p, p, p, p, 1, 32, 65536, 65536, 128, 0.088, 1, 8, p, p, p, p,
                                  None)
    assert st == binding.STREAMKL_ERR_INVALID_ARG
    msg = lib.streamkl_last_error()
    assert str(SCRATCH_BYTES).encode() in msg and b"workspace" in msg


def _close(got, ref):
    err = (got.double() - ref.double()).abs()
    bound = KL_ABS + KL_REL * ref.double().abs()
    return bool((err <= bound).all())


def _rel_l2(got, ref):
    return float((got.double() - ref.double()).norm() / ref.double().norm())


@pytest.mark.gpu
def test_noalloc_forward_matches_workspace_forward_on_two_calls(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    cases = [
        (synthetic.custom("noalloc_a", B=2, H=4, NQ=384, NK=4096 + 77, d=128, causal=True,
                          noise=0.2), 4, 11),
        (synthetic.custom("noalloc_b", B=1, H=8, NQ=200, NK=3000, d=64, causal=False,
                          teacher_std=2.0, noise=0.5), 3, 12),
    ]
    for w, splits, seed in cases:
        assert binding.streamkl_fwd_workspace_size(w.B, w.H, w.NQ, w.NK, w.d, w.causal,
                                                   splits) > 0  # the scratch is really used
        q1, k1, q2, k2, _ = synthetic.make_inputs(w, seed, dev)
        ref = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, num_splits=splits)
        out = tuple(torch.full((w.B, w.H, w.NQ), float("nan"), device=dev) for _ in range(3))
        status = binding.new_status(dev)
        binding.streamkl_fwd_noalloc(q1, k1, q2, k2, out, w.scale, w.causal, num_splits=splits,
                                     dev_status=status)
        binding.raise_on_device_status(status, "streamkl_fwd_noalloc")
        kl, lse1, lse2 = out
        assert torch.isfinite(kl).all()
        assert _close(kl, ref[0]), w.name
        assert _rel_l2(lse1, ref[1]) <= LSE_REL
        assert _rel_l2(lse2, ref[2]) <= LSE_REL
    assert np.isfinite(float(kl.sum()))


@pytest.mark.gpu
def test_noalloc_automatic_split_against_the_oracle(lib):
    """num_splits = 0 (the library's own split choice, the normal way to call
    it) on a decode-like shape where that choice splits the keys, so the
    built-in scratch is used; outputs against the fp64 oracle and against the
    workspace forward."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    w = synthetic.custom("noalloc_decode", B=1, H=4, NQ=64, NK=65536, d=128, causal=True,
                         noise=0.3)
    splits = binding.choose_splits(w.B, w.H, w.NQ, w.NK, w.d, w.causal)
    assert splits > 1
    assert 0 < binding.streamkl_fwd_workspace_size(w.B, w.H, w.NQ, w.NK, w.d, w.causal,
                                                   0) <= SCRATCH_BYTES
    q1, k1, q2, k2, _ = synthetic.make_inputs(w, 13, dev)
    out = tuple(torch.full((w.B, w.H, w.NQ), float("nan"), device=dev) for _ in range(3))
    status = binding.new_status(dev)
    binding.streamkl_fwd_noalloc(q1, k1, q2, k2, out, w.scale, w.causal, num_splits=0,
                                 dev_status=status)
    binding.raise_on_device_status(status, "streamkl_fwd_noalloc")
    ref = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, num_splits=0)
    kl, lse1, lse2 = out
    assert _close(kl, ref[0])
    h = [t.float().cpu().numpy().astype(np.float64) for t in (q1, k1, q2, k2)]
    okl, ol1, ol2 = orc.forward(*h, w.scale, w.causal)
    err = np.abs(kl.cpu().numpy().astype(np.float64) - okl)
    assert np.all(err <= KL_ABS + KL_REL * np.abs(okl))
    for got, want in ((lse1, ol1), (lse2, ol2)):
        g = got.cpu().numpy().astype(np.float64)
        assert np.linalg.norm(g - want) / np.linalg.norm(want) <= LSE_REL
