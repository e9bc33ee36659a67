"""The C-ABI calls inside a CUDA graph: the library only enqueues work on the
caller's stream (no allocation, no synchronisation), so a forward + backward
step captured once replays with results identical to eager calls, including
after new inputs are copied into the captured buffers."""
import pytest
import torch

from attention_kl_loss_gb300 import binding, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


@pytest.mark.parametrize("NQ,NK,d,causal,grad1", [(384, 640, 128, True, True),
                                                   (256, 8192, 64, True, False)])
def test_captured_step_replays_like_eager(NQ, NK, d, causal, grad1):
    w = synthetic.custom(f"graph_{NQ}x{NK}d{d}", B=1, H=4, NQ=NQ, NK=NK, d=d, causal=causal,
                         noise=0.3, grad1=grad1)
    dev = torch.device("cuda")
    static = [t.clone() for t in synthetic.make_inputs(w, 1, dev)]
    q1, k1, q2, k2, g = static
    B, H = w.B, w.H
    ws = torch.empty(max(binding.streamkl_workspace_size(B, H, NQ, NK, d, causal, grad1), 256),
                     dtype=torch.uint8, device=dev)
    status = binding.new_status(dev)
    outs = tuple(torch.empty((B, H, NQ), device=dev) for _ in range(3))
    grads = (torch.empty_like(q2), torch.empty_like(k2),
             torch.empty_like(q1) if grad1 else None, torch.empty_like(k1) if grad1 else None)

    def step():
        kl, l1, l2 = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, causal, out=outs,
                                          workspace=ws, dev_status=status)
        binding.streamkl_bwd(q1, k1, q2, k2, kl, l1, l2, g, w.scale, causal, grad1=grad1,
                             out=grads, workspace=ws, dev_status=status)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside the capture (attributes, tensor-map encoder)
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for seed in (2, 3):
        for dst, src in zip(static, synthetic.make_inputs(w, seed, dev)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in outs] + [t.clone() for t in grads if t is not None]
        step()  # eager, same buffers
        torch.cuda.synchronize()
        ref = list(outs) + [t for t in grads if t is not None]
        binding.raise_on_device_status(status, "graph replay")
        for a, b in zip(got, ref):
            assert torch.equal(a, b)


# (name, shape): separate kernels, split forward with a workspace, the
# short-sweep fused backward and the fused d = 64 backward (their dQ summed
# with fp32 reductions)
CASES = [
    ("separate", dict(B=2, H=3, NQ=300, NK=333, d=128, causal=True, grad1=True)),
    ("split forward d64", dict(B=1, H=4, NQ=64, NK=8192, d=64, causal=True)),
    ("short sweep", dict(B=2, H=8, NQ=48, NK=4000, d=128, causal=True, grad1=True)),
    ("fused d64", dict(B=1, H=2, NQ=640, NK=700, d=64, causal=True)),
    ("fused d128", dict(B=1, H=2, NQ=600, NK=650, d=128, causal=False)),
]


def _step(w, ins, status):
    q1, k1, q2, k2, g = ins
    out = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, dev_status=status)
    grads = binding.streamkl_bwd(q1, k1, q2, k2, *out, g, w.scale, w.causal, grad1=w.grad1,
                                 dev_status=status)
    return tuple(out) + tuple(grads)


def _close(got, want, what, atomic_dq):
    for i, (x, y) in enumerate(zip(got, want)):
        assert (x is None) == (y is None), (what, i)
        if x is None:
            continue
        if atomic_dq and i in (3, 5):
            err = (x.double() - y.double()).norm() / max(float(y.double().norm()), 1e-30)
            assert float(err) <= 1e-3, (what, i, float(err))
        else:
            assert torch.equal(x, y), (what, i)


@pytest.mark.parametrize("name,shape", CASES, ids=[c[0] for c in CASES])
def test_captured_step_with_binding_allocations(name, shape):
    """Outputs and workspace allocated by the binding inside the capture (from
    the graph's memory pool), on the separate, split-forward, short-sweep and
    per-key-tile fused paths; the fused paths sum dQ with fp32 reductions, so
    it matches to rounding."""
    w = synthetic.custom(name.replace(" ", "_"), noise=0.3, **shape)
    dev = torch.device("cuda")
    ins = synthetic.make_inputs(w, 41, dev)
    status = binding.new_status(dev)
    fused = binding.bwd_algorithm(w.B, w.H, w.NQ, w.NK, w.d, w.causal, w.grad1) == binding.BWD_FUSED
    if name == "split forward d64":
        assert binding.choose_splits(w.B, w.H, w.NQ, w.NK, w.d, w.causal) > 1
    if name.startswith("fused"):
        assert fused

    eager = _step(w, ins, status)  # also loads every kernel before the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = _step(w, ins, status)
    graph.replay()
    torch.cuda.synchronize()
    binding.raise_on_device_status(status, name)
    _close(captured, eager, f"{name}: replay", fused)

    # new values in the same buffers: the replay reads them
    fresh = synthetic.make_inputs(w, 42, dev)
    for dst, src in zip(ins, fresh):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    again = _step(w, ins, status)
    torch.cuda.synchronize()
    binding.raise_on_device_status(status, name)
    _close(captured, again, f"{name}: replay on new inputs", fused)
    assert not torch.equal(captured[0], eager[0])
