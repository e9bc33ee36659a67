"""Packed variable-length batches through the C ABI against the fp64 oracle,
one (sequence, head) slice at a time (heads and sequences are independent).
Tolerances as in test_gpu_parity.py."""
import numpy as np
import pytest
import torch

from attention_kl_loss_gb300 import binding, synthetic
from oracle import streamkl_oracle as orc

pytestmark = pytest.mark.gpu

KL_ABS, KL_REL, LSE_REL, GRAD_REL = 2e-3, 1e-2, 1e-4, 1e-2


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _rel_l2(got, ref):
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def _run(lens_q, lens_k, H, d, causal, seed=5, grad1=True, grad2=True):
    dev = torch.device("cuda")
    q1, k1, q2, k2, g, cu_q, cu_k = synthetic.make_packed_inputs(lens_q, lens_k, H, d, seed,
                                                                 device=dev)
    st = binding.new_status(dev)
    mq, mk = max(lens_q), max(lens_k)
    scale = d ** -0.5
    kl, l1, l2 = binding.streamkl_fwd_varlen(q1, k1, q2, k2, cu_q, cu_k, mq, mk, scale, causal,
                                             dev_status=st)
    grads = binding.streamkl_bwd_varlen(q1, k1, q2, k2, cu_q, cu_k, mq, mk, kl, l1, l2, g, scale,
                                        causal, grad1=grad1, grad2=grad2, dev_status=st)
    torch.cuda.synchronize()
    return (q1, k1, q2, k2, g, cu_q.tolist(), cu_k.tolist(), scale), (kl, l1, l2), grads, st


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_batch_matches_oracle_per_sequence(d, causal):
    lens_q = [100, 300, 0, 1, 129]
    lens_k = [150, 300, 7, 64, 200]
    ins, (kl, l1, l2), grads, st = _run(lens_q, lens_k, 2, d, causal)
    assert int(st.item()) == 0
    q1, k1, q2, k2, g, cu_q, cu_k, scale = ins
    for b in range(len(lens_q)):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe == qs:
            # no query sees this sequence's keys: their gradients are exactly 0
            for t in (grads[1], grads[3]):
                assert torch.all(t[ks:ke].float() == 0), b
            continue
        for h in range(2):
            sl = [_f64(t[a:e, h]) for t, a, e in ((q1, qs, qe), (k1, ks, ke), (q2, qs, qe),
                                                  (k2, ks, ke))]
            okl, ol1, ol2 = orc.head_forward(*sl, scale, causal)
            err = np.abs(kl[qs:qe, h].cpu().numpy() - okl)
            assert np.all(err <= KL_ABS + KL_REL * np.abs(okl)), (b, h, float(err.max()))
            assert _rel_l2(l1[qs:qe, h].cpu().numpy(), ol1) <= LSE_REL
            assert _rel_l2(l2[qs:qe, h].cpu().numpy(), ol2) <= LSE_REL
            og = orc.head_backward(*sl, scale, causal, _f64(g[qs:qe, h]), True)
            for got, ref, name in ((grads[0][qs:qe, h], og[0], "dq2"), (grads[1][ks:ke, h], og[1], "dk2"),
                                   (grads[2][qs:qe, h], og[2], "dq1"), (grads[3][ks:ke, h], og[3], "dk1")):
                got = _f64(got)
                if not np.any(ref):
                    assert np.max(np.abs(got)) <= 1e-5, (b, h, name)
                else:
                    assert _rel_l2(got, ref) <= GRAD_REL, (b, h, name, _rel_l2(got, ref))


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
@pytest.mark.parametrize("sets", ["config1", "config2"])
def test_packed_batch_one_gradient_set(sets, d, causal):
    """Either configuration alone on a packed batch: the requested pair
    against the oracle, the other pair not produced."""
    lens_q, lens_k = [70, 0, 257, 3], [90, 5, 300, 64]
    grad1, grad2 = sets == "config2", sets == "config1"
    ins, (kl, l1, l2), grads, st = _run(lens_q, lens_k, 2, d, causal, seed=8, grad1=grad1,
                                        grad2=grad2)
    assert int(st.item()) == 0
    assert (grads[0] is None) == (not grad2) and (grads[2] is None) == (not grad1)
    q1, k1, q2, k2, g, cu_q, cu_k, scale = ins
    for b in range(len(lens_q)):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        for h in range(2):
            if qe == qs:
                for t in (grads[1], grads[3]):
                    if t is not None:
                        assert torch.all(t[ks:ke, h].float() == 0), b
                continue
            sl = [_f64(t[a:e, h]) for t, a, e in ((q1, qs, qe), (k1, ks, ke), (q2, qs, qe),
                                                  (k2, ks, ke))]
            og = orc.head_backward(*sl, scale, causal, _f64(g[qs:qe, h]), True)
            for i, (lo, hi) in enumerate(((qs, qe), (ks, ke), (qs, qe), (ks, ke))):
                if grads[i] is None:
                    continue
                got, ref = _f64(grads[i][lo:hi, h]), og[i]
                if not np.any(ref):
                    assert np.max(np.abs(got)) <= 1e-5, (b, h, i)
                else:
                    assert _rel_l2(got, ref) <= GRAD_REL, (b, h, i, _rel_l2(got, ref))


def test_single_sequence_equals_dense_api():
    """One sequence packed [N, H, d] is the dense [1, H, N, d] problem."""
    n, h, d = 384, 3, 128
    ins, (kl, l1, l2), grads, st = _run([n], [n], h, d, True, seed=9)
    assert int(st.item()) == 0
    q1, k1, q2, k2, g = (t.transpose(0, 1).unsqueeze(0).contiguous() for t in ins[:5])
    ref = binding.streamkl_fwd(q1, k1, q2, k2, ins[7], True, num_splits=1)
    assert torch.allclose(kl.t().unsqueeze(0), ref[0], rtol=1e-5, atol=1e-6)
    rg = binding.streamkl_bwd(q1, k1, q2, k2, *ref, g, ins[7], True, grad1=True)
    for got, want in zip(grads, rg):
        assert torch.equal(got.transpose(0, 1).unsqueeze(0), want)


def test_device_checks_of_the_offsets():
    """A causal sequence with more query rows than keys is reported through
    the status word (the kernels return normally; what they computed is not
    to be used)."""
    _, _, _, st = _run([50, 200], [80, 100], 2, 64, True, seed=3)
    assert int(st.item()) == binding.STREAMKL_ERR_INVALID_ARG


def test_sequence_with_queries_but_no_keys_is_reported():
    """Query rows with no key at all (non-causal) have no softmax: the forward
    reports STREAMKL_ERR_INVALID_ARG through the status word."""
    dev = torch.device("cuda")
    lens_q, lens_k = [40, 30], [0, 90]
    q1, k1, q2, k2, g, cu_q, cu_k = synthetic.make_packed_inputs(lens_q, lens_k, 2, 64, 4,
                                                                 device=dev)
    st = binding.new_status(dev)
    binding.streamkl_fwd_varlen(q1, k1, q2, k2, cu_q, cu_k, max(lens_q), max(lens_k), None, False,
                                dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == binding.STREAMKL_ERR_INVALID_ARG
