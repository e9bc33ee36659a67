"""The debug build (libstreamkl_debug.so, compiled with STREAMKL_DEVICE_CHECKS)
on the GPU: every TMA copy, TMEM access and mbarrier of every kernel is
range-checked before it is issued. On the small parity shapes, through every
kernel variant (split forward, both backward algorithms, the dQ key split,
the persistent dK kernel, packed batches), no check may fail (the status
word stays 0) and the results must equal the release build's bit for bit:
the checks add branches, never arithmetic. The report path itself is
exercised by a self-test kernel that checks a range past any allocation
without touching it."""
import pytest
import torch

from attention_kl_loss_gb300 import binding, build, synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _libs(cuda_lib):
    build.build(debug=True)
    return binding.load(debug=True)


def test_check_selftest_reports_only_in_the_debug_build():
    st = binding.selftest_device_check()
    torch.cuda.synchronize()
    assert int(st.item()) == 0  # release build: checks compiled out
    with binding.use_debug_library():
        st = binding.selftest_device_check()
        torch.cuda.synchronize()
    assert int(st.item()) == binding.STREAMKL_ERR_DEVICE_CHECK
    x = torch.ones(4, device="cuda")  # the context is still usable
    assert float(x.sum().item()) == 4.0


def _dense_run(w, seed, splits=0, algo=None, dq_splits=None, dk_persist=None, grad2=True,
               pairs=None):
    dev = torch.device("cuda")
    q1, k1, q2, k2, g = synthetic.make_inputs(w, seed, dev)
    st = binding.new_status(dev)
    binding.set_bwd_algorithm(algo)
    binding.set_bwd_dq_splits(dq_splits)
    binding.set_bwd_dk_persist(dk_persist)
    binding.set_fwd_pairs(pairs)
    try:
        kl, l1, l2 = binding.streamkl_fwd(q1, k1, q2, k2, w.scale, w.causal, num_splits=splits,
                                          dev_status=st)
        grads = binding.streamkl_bwd(q1, k1, q2, k2, kl, l1, l2, g, w.scale, w.causal,
                                     grad1=w.grad1, grad2=grad2, dev_status=st)
    finally:
        binding.set_bwd_algorithm(None)
        binding.set_bwd_dq_splits(None)
        binding.set_bwd_dk_persist(None)
        binding.set_fwd_pairs(None)
    binding.raise_on_device_status(st, w.name)
    return (kl, l1, l2) + tuple(grads)


def _same(a, b, what, atomic_dq=False):
    """Bit-equal, except the dQ of the fused algorithm (outputs 3 and 5): it
    is summed with fp32 global reductions whose order differs from run to
    run, so two runs of the same build agree only to rounding."""
    for i, (x, y) in enumerate(zip(a, b)):
        assert (x is None) == (y is None), (what, i)
        if x is None:
            continue
        if atomic_dq and i in (3, 5):
            err = (x.double() - y.double()).norm() / max(float(y.double().norm()), 1e-30)
            assert float(err) <= 1e-3, (what, i, float(err))
        else:
            assert torch.equal(x, y), (what, i)


CASES = [
    ("tiny both sets", dict(B=1, H=2, NQ=256, NK=256, d=64, causal=False, grad1=True), {}),
    ("ragged causal d128", dict(B=2, H=3, NQ=200, NK=333, d=128, causal=True, grad1=True), {}),
    ("ragged d64 one set", dict(B=2, H=3, NQ=333, NK=200, d=64, causal=False, grad1=False), {}),
    ("one row", dict(B=1, H=2, NQ=1, NK=300, d=128, causal=True, grad1=True), {}),
    ("forced split forward", dict(B=1, H=4, NQ=256, NK=2125, d=128, causal=True), {"splits": 3}),
    ("fused backward", dict(B=2, H=3, NQ=200, NK=333, d=128, causal=True, grad1=True),
     {"algo": binding.BWD_FUSED}),
    ("fused backward d64", dict(B=1, H=2, NQ=130, NK=131, d=64, causal=True, grad1=False),
     {"algo": binding.BWD_FUSED}),
    ("dQ key split", dict(B=1, H=2, NQ=200, NK=2000, d=128, causal=True, grad1=True),
     {"algo": binding.BWD_SEPARATE, "dq_splits": 3}),
    ("persistent dK", dict(B=2, H=2, NQ=64, NK=4096, d=128, causal=True), {"dk_persist": 3}),
    ("configuration 2 only", dict(B=2, H=3, NQ=130, NK=131, d=64, causal=True, grad1=True),
     {"grad2": False}),
    ("short sweep both sets", dict(B=4, H=10, NQ=20, NK=1000, d=128, causal=True, grad1=True), {}),
    ("short sweep one set", dict(B=2, H=3, NQ=64, NK=777, d=128, causal=False), {}),
    ("short sweep configuration 2 only", dict(B=2, H=3, NQ=48, NK=2000, d=128, causal=True,
                                               grad1=True), {"grad2": False}),
    ("forward as CTA pairs", dict(B=2, H=3, NQ=256, NK=333, d=128, causal=True),
     {"splits": 1, "pairs": True}),
    ("forward as CTA pairs d64", dict(B=1, H=4, NQ=200, NK=200, d=64, causal=True),
     {"splits": 1, "pairs": True}),
]


@pytest.mark.parametrize("name,shape,opts", CASES, ids=[c[0] for c in CASES])
def test_debug_build_passes_its_checks_and_matches_release(name, shape, opts):
    w = synthetic.custom(name.replace(" ", "_"), noise=0.4, **shape)
    ref = _dense_run(w, 31, **opts)
    with binding.use_debug_library():
        got = _dense_run(w, 31, **opts)
    fused = opts.get("algo", binding.bwd_algorithm(w.B, w.H, w.NQ, w.NK, w.d, w.causal,
                                                  w.grad1)) == binding.BWD_FUSED
    _same(got, ref, name, atomic_dq=fused)


@pytest.mark.parametrize("causal", [False, True])
def test_debug_build_packed_batches(causal):
    dev = torch.device("cuda")
    lens_q, lens_k = [100, 300, 0, 1, 129], [150, 300, 7, 64, 200]
    q1, k1, q2, k2, g, cu_q, cu_k = synthetic.make_packed_inputs(lens_q, lens_k, 2, 128, 9,
                                                                 device=dev)
    mq, mk = max(lens_q), max(lens_k)

    def run():
        st = binding.new_status(dev)
        out = binding.streamkl_fwd_varlen(q1, k1, q2, k2, cu_q, cu_k, mq, mk, None, causal,
                                          dev_status=st)
        grads = binding.streamkl_bwd_varlen(q1, k1, q2, k2, cu_q, cu_k, mq, mk, *out, g, None,
                                            causal, grad1=True, dev_status=st)
        binding.raise_on_device_status(st, "packed")
        return tuple(out) + tuple(grads)

    ref = run()
    with binding.use_debug_library():
        got = run()
    _same(got, ref, "packed")
