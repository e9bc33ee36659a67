"""Pins for the fp64 oracle: each check comes from outside the oracle itself.

Sources of truth used here (none re-types the oracle's own formula):
* library routines: scipy.stats.entropy (KL of two discrete distributions),
  scipy.special.logsumexp / softmax, torch autograd through log_softmax;
* closed forms: Bernoulli KL for two keys, log N_K for a one-hot teacher
  against a uniform student, hand-worked 2-key cases;
* invariants: KL = 0 for identical inputs, KL >= 0 (Gibbs), shift invariance
  of softmax along keys, causal == truncated non-causal, head independence;
* brute force: pure-Python loops on tiny inputs; central finite differences.
The last test plants mistakes in the oracle and checks that a pin catches
each one.
"""
import math

import numpy as np
import pytest
import scipy.special as sps
import scipy.stats as sst
import torch

from oracle import streamkl_oracle as orc


def _rand(rng, *shape, std=1.0):
    return rng.standard_normal(shape) * std


def _case(seed, n_q, n_k, d, std=1.0, noise=0.5):
    rng = np.random.default_rng(seed)
    q1 = _rand(rng, n_q, d, std=std)
    k1 = _rand(rng, n_k, d, std=std)
    q2 = q1 + _rand(rng, n_q, d, std=noise)
    k2 = k1 + _rand(rng, n_k, d, std=noise)
    return q1, k1, q2, k2


SHAPES = [(1, 1, 4, False), (5, 7, 4, False), (7, 7, 8, True), (5, 9, 8, True),
          (33, 70, 16, True), (64, 64, 32, False), (300, 300, 16, True)]


@pytest.mark.parametrize("n_q,n_k,d,causal", SHAPES)
def test_forward_matches_scipy(n_q, n_k, d, causal):
    """KL per row == scipy.stats.entropy(P1, P2); lse == scipy logsumexp."""
    q1, k1, q2, k2 = _case(1, n_q, n_k, d)
    scale = 1 / math.sqrt(d)
    kl, lse1, lse2 = orc.head_forward(q1, k1, q2, k2, scale, causal)
    for i in range(n_q):
        n = n_k if not causal else i + 1 + (n_k - n_q)
        s1 = scale * (q1[i] @ k1[:n].T)
        s2 = scale * (q2[i] @ k2[:n].T)
        p1, p2 = sps.softmax(s1), sps.softmax(s2)
        assert kl[i] == pytest.approx(sst.entropy(p1, p2), rel=1e-10, abs=1e-13)
        assert lse1[i] == pytest.approx(sps.logsumexp(s1), rel=1e-13)
        assert lse2[i] == pytest.approx(sps.logsumexp(s2), rel=1e-13)


def test_bruteforce_python_loops():
    """Pure-Python triple loop with math.exp/math.log on a tiny causal case."""
    n_q, n_k, d = 3, 5, 2
    q1, k1, q2, k2 = _case(7, n_q, n_k, d)
    scale = 0.7
    kl, _, _ = orc.head_forward(q1, k1, q2, k2, scale, True)
    for i in range(n_q):
        keys = range(i + 1 + (n_k - n_q))
        s1 = [scale * sum(q1[i][c] * k1[j][c] for c in range(d)) for j in keys]
        s2 = [scale * sum(q2[i][c] * k2[j][c] for c in range(d)) for j in keys]
        z1 = sum(math.exp(v) for v in s1)
        z2 = sum(math.exp(v) for v in s2)
        ref = sum(math.exp(a) / z1 * math.log((math.exp(a) / z1) / (math.exp(b) / z2))
                  for a, b in zip(s1, s2))
        assert kl[i] == pytest.approx(ref, rel=1e-12, abs=1e-15)


def test_hand_worked_two_keys():
    """s1 = (ln 3, 0), s2 = (0, 0): P1 = (3/4, 1/4), P2 = (1/2, 1/2).

    KL = 3/4 ln(3/2) + 1/4 ln(1/2); lse1 = ln 4; lse2 = ln 2.
    Gradient of KL w.r.t. s2 is P2 - P1 = (-1/4, 1/4), so with k2 = (1, 0)^T
    rows, dq2 = -1/4 (scale 1, g 1); w.r.t. s1 it is
    P1 * (log(P1/P2) - KL), which with k1 rows (1, 0) gives
    dq1 = 3/4 (ln(3/2) - KL).
    """
    q1 = np.array([[math.log(3.0)]])
    k1 = np.array([[1.0], [0.0]])
    q2 = np.array([[0.0]])
    k2 = np.array([[1.0], [0.0]])
    kl, lse1, lse2 = orc.head_forward(q1, k1, q2, k2, 1.0, False)
    want = 0.75 * math.log(1.5) + 0.25 * math.log(0.5)
    assert kl[0] == pytest.approx(want, rel=1e-14)
    assert lse1[0] == pytest.approx(math.log(4.0), rel=1e-14)
    assert lse2[0] == pytest.approx(math.log(2.0), rel=1e-14)
    dq2, dk2, dq1, dk1 = orc.head_backward(q1, k1, q2, k2, 1.0, False, np.ones(1), True)
    assert dq2[0, 0] == pytest.approx(-0.25, rel=1e-14)
    # dk2[j] = dS2[j] * q2 = 0 because q2 = 0
    assert np.all(dk2 == 0)
    assert dq1[0, 0] == pytest.approx(0.75 * (math.log(1.5) - want), rel=1e-13)
    # dk1[j] = dS1[j] * q1; dS1 = P1 (log(P1/P2) - KL)
    ds1 = np.array([0.75 * (math.log(1.5) - want), 0.25 * (math.log(0.5) - want)])
    assert dk1[:, 0] == pytest.approx(ds1 * math.log(3.0), rel=1e-13)


@pytest.mark.parametrize("n_q,n_k,d,causal", SHAPES)
@pytest.mark.parametrize("tiles", [(1,), (3,), (16,), (5, 2, 11), (64,), (1000,)])
def test_online_form_equals_two_pass(n_q, n_k, d, causal, tiles):
    """The pages' five-scalar streaming update reproduces the definition."""
    q1, k1, q2, k2 = _case(3, n_q, n_k, d, std=2.0, noise=1.0)
    scale = 1 / math.sqrt(d)
    a = orc.head_forward(q1, k1, q2, k2, scale, causal)
    b = orc.head_forward_online(q1, k1, q2, k2, scale, causal, tiles)
    for x, y in zip(a, b):
        np.testing.assert_allclose(y, x, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_inputs_give_zero(causal):
    q, k, _, _ = _case(5, 40, 64, 8)
    kl, lse1, lse2 = orc.head_forward(q, k, q, k, 0.3, causal)
    assert np.all(kl == 0.0)
    assert np.all(lse1 == lse2)
    grads = orc.head_backward(q, k, q, k, 0.3, causal, np.full(40, 0.1), True)
    for gr in grads:
        assert np.all(gr == 0.0)


@pytest.mark.parametrize("seed", range(5))
def test_kl_nonnegative(seed):
    q1, k1, q2, k2 = _case(seed, 50, 80, 16, std=3.0, noise=2.0)
    kl, _, _ = orc.head_forward(q1, k1, q2, k2, 0.25, seed % 2 == 1)
    assert np.all(kl >= -1e-15)
    assert np.any(kl > 1e-3)


@pytest.mark.parametrize("causal,n_q,n_k", [(False, 6, 9), (True, 6, 9), (True, 8, 8)])
def test_one_hot_teacher_vs_uniform_student(causal, n_q, n_k):
    """K2 = 0 makes P2 uniform over the allowed keys; a teacher with one key far
    ahead is one-hot, so KL = log(#allowed keys) (within exp(-gap))."""
    d, gap = 3, 60.0
    q1 = np.zeros((n_q, d))
    q1[:, 0] = gap
    k1 = np.zeros((n_k, d))
    k1[0, 0] = 1.0  # key 0 is allowed for every row, even under causal masking
    q2 = np.ones((n_q, d))
    k2 = np.zeros((n_k, d))
    kl, _, lse2 = orc.head_forward(q1, k1, q2, k2, 1.0, causal)
    for i in range(n_q):
        n = n_k if not causal else i + 1 + (n_k - n_q)
        assert kl[i] == pytest.approx(math.log(n), abs=1e-20 + n * math.exp(-gap) * gap)
        assert lse2[i] == pytest.approx(math.log(n), rel=1e-14)


def test_uniform_student_general_teacher():
    """With P2 uniform, KL = log N_K - H(P1) with H the Shannon entropy."""
    q1, k1, _, _ = _case(11, 10, 23, 6, std=1.5)
    q2 = np.ones((10, 6))
    k2 = np.zeros((23, 6))
    kl, _, _ = orc.head_forward(q1, k1, q2, k2, 0.5, False)
    for i in range(10):
        p1 = sps.softmax(0.5 * q1[i] @ k1.T)
        assert kl[i] == pytest.approx(math.log(23) - sst.entropy(p1), rel=1e-11)


def test_two_keys_bernoulli():
    """N_K = 2: KL is the Bernoulli KL of sigmoid(s_0 - s_1)."""
    q1, k1, q2, k2 = _case(13, 9, 2, 5, std=1.3)
    kl, _, _ = orc.head_forward(q1, k1, q2, k2, 0.8, False)
    for i in range(9):
        s1 = 0.8 * q1[i] @ k1.T
        s2 = 0.8 * q2[i] @ k2.T
        p = sps.expit(s1[0] - s1[1])
        q = sps.expit(s2[0] - s2[1])
        want = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
        assert kl[i] == pytest.approx(want, rel=1e-11, abs=1e-15)


@pytest.mark.parametrize("which", ["k1", "k2"])
def test_shift_invariance_along_keys(which):
    """Adding one vector c to every key shifts a row's logits by a constant:
    KL and the gradients are unchanged, and sum_j dK_t[j] = 0."""
    q1, k1, q2, k2 = _case(17, 12, 20, 8)
    c = np.random.default_rng(2).standard_normal(8)
    g = np.random.default_rng(3).random(12)
    base_f = orc.head_forward(q1, k1, q2, k2, 0.4, True)
    base_b = orc.head_backward(q1, k1, q2, k2, 0.4, True, g, True)
    if which == "k1":
        k1 = k1 + c
    else:
        k2 = k2 + c
    f = orc.head_forward(q1, k1, q2, k2, 0.4, True)
    b = orc.head_backward(q1, k1, q2, k2, 0.4, True, g, True)
    np.testing.assert_allclose(f[0], base_f[0], rtol=1e-10, atol=1e-13)
    for x, y in zip(b, base_b):
        np.testing.assert_allclose(x, y, rtol=1e-9, atol=1e-13)
    for dk in (b[1], b[3]):
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-13)


def test_causal_equals_truncated_noncausal():
    """Causal row i (bottom-right) == non-causal over keys 0..i+N_K-N_Q."""
    n_q, n_k = 9, 14
    q1, k1, q2, k2 = _case(19, n_q, n_k, 4)
    kl, lse1, lse2 = orc.head_forward(q1, k1, q2, k2, 0.6, True)
    for i in range(n_q):
        n = i + 1 + (n_k - n_q)
        a = orc.head_forward(q1[i:i + 1], k1[:n], q2[i:i + 1], k2[:n], 0.6, False)
        assert (kl[i], lse1[i], lse2[i]) == pytest.approx(tuple(x[0] for x in a), rel=1e-13)


def test_head_independence():
    rng = np.random.default_rng(23)
    x = [rng.standard_normal((2, 3, 6, 4)) for _ in range(4)]
    kl_a, _, _ = orc.forward(*x, 0.5, False)
    y = [t.copy() for t in x]
    for t in y:
        t[1, 2] += 5 * rng.standard_normal(t[1, 2].shape)
    kl_b, _, _ = orc.forward(*y, 0.5, False)
    mask = np.ones((2, 3), bool)
    mask[1, 2] = False
    np.testing.assert_array_equal(kl_a[mask], kl_b[mask])
    assert not np.allclose(kl_a[1, 2], kl_b[1, 2])


def _loss(q1, k1, q2, k2, scale, causal, g):
    kl, _, _ = orc.head_forward(q1, k1, q2, k2, scale, causal)
    return float(np.dot(g, kl))


def _fd_check(n_q, n_k, d, causal, seed, tol=1e-6):
    q1, k1, q2, k2 = _case(seed, n_q, n_k, d, std=1.2, noise=0.8)
    g = np.random.default_rng(seed + 100).random(n_q) + 0.5
    scale = 0.45
    dq2, dk2, dq1, dk1 = orc.head_backward(q1, k1, q2, k2, scale, causal, g, True)
    h = 1e-5
    args = [q1, k1, q2, k2]
    for idx, grad in [(0, dq1), (1, dk1), (2, dq2), (3, dk2)]:
        fd = np.zeros_like(args[idx])
        for e in np.ndindex(fd.shape):
            a = [t.copy() for t in args]
            a[idx][e] += h
            lp = _loss(*a, scale, causal, g)
            a[idx][e] -= 2 * h
            lm = _loss(*a, scale, causal, g)
            fd[e] = (lp - lm) / (2 * h)
        err = np.max(np.abs(fd - grad)) / max(np.max(np.abs(fd)), 1e-30)
        assert err < tol, (idx, err)


@pytest.mark.parametrize("n_q,n_k,d,causal", [(5, 7, 4, False), (5, 7, 4, True),
                                               (7, 7, 8, True), (16, 16, 4, False)])
def test_gradients_central_finite_differences(n_q, n_k, d, causal):
    _fd_check(n_q, n_k, d, causal, seed=n_q * 31 + n_k)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd(causal):
    """Independent route: torch fp64 autograd through log_softmax/kl_div."""
    n_q, n_k, d = 11, 17, 8
    q1, k1, q2, k2 = _case(29, n_q, n_k, d, std=1.5, noise=0.7)
    g = np.random.default_rng(31).random(n_q)
    scale = 0.35
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q1, k1, q2, k2)]
    rows = []
    for i in range(n_q):
        n = n_k if not causal else i + 1 + (n_k - n_q)  # allowed keys, sliced not masked
        lp1 = torch.log_softmax(scale * t[1][:n] @ t[0][i], dim=-1)
        lp2 = torch.log_softmax(scale * t[3][:n] @ t[2][i], dim=-1)
        rows.append(torch.nn.functional.kl_div(lp2, lp1, reduction="sum", log_target=True))
    kl = torch.stack(rows)
    (kl * torch.tensor(g)).sum().backward()
    ours = orc.head_backward(q1, k1, q2, k2, scale, causal, g, True)
    kl_o, _, _ = orc.head_forward(q1, k1, q2, k2, scale, causal)
    np.testing.assert_allclose(kl_o, kl.detach().numpy(), rtol=1e-11, atol=1e-14)
    for ref, got in [(t[2].grad, ours[0]), (t[3].grad, ours[1]), (t[0].grad, ours[2]),
                     (t[1].grad, ours[3])]:
        np.testing.assert_allclose(got, ref.numpy(), rtol=1e-9, atol=1e-13)


def test_row_subset_backward_is_partial_sum():
    """head_backward over a row subset returns those rows' dQ and their dK
    contributions; the subsets add up to the full result."""
    q1, k1, q2, k2 = _case(37, 20, 20, 4)
    g = np.linspace(0.5, 1.5, 20)
    full = orc.head_backward(q1, k1, q2, k2, 0.5, True, g, True)
    a = orc.head_backward(q1, k1, q2, k2, 0.5, True, g, True, rows=np.arange(0, 7))
    b = orc.head_backward(q1, k1, q2, k2, 0.5, True, g, True, rows=np.arange(7, 20))
    np.testing.assert_allclose(np.concatenate([a[0], b[0]]), full[0], rtol=1e-13)
    np.testing.assert_allclose(a[1] + b[1], full[1], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(a[3] + b[3], full[3], rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("mutation", ["ds1_drop_kl", "ds2_sign", "ds1_no_p1"])
def test_planted_mistakes_are_caught(monkeypatch, mutation):
    """Plant a plausible slip in the oracle's Jacobian; the finite-difference
    pin must fail on it."""
    if mutation == "ds1_drop_kl":
        monkeypatch.setattr(orc, "dkl_ds1", lambda p1, lr, kl: p1 * lr)
    elif mutation == "ds2_sign":
        monkeypatch.setattr(orc, "dkl_ds2", lambda p1, p2: p1 - p2)
    else:
        monkeypatch.setattr(orc, "dkl_ds1", lambda p1, lr, kl: lr - kl[:, None])
    with pytest.raises(AssertionError):
        _fd_check(5, 7, 4, True, seed=3)


def _batched_case():
    """B = 2, H = 3, N_Q != N_K, four distinct tensors, g varying per (b, h, row)."""
    rng = np.random.default_rng(41)
    B, H, n_q, n_k, d = 2, 3, 6, 9, 5
    q1 = rng.standard_normal((B, H, n_q, d)) * 1.3
    k1 = rng.standard_normal((B, H, n_k, d)) * 1.1
    q2 = rng.standard_normal((B, H, n_q, d)) * 0.9
    k2 = rng.standard_normal((B, H, n_k, d)) * 1.2
    g = rng.standard_normal((B, H, n_q))
    return q1, k1, q2, k2, g, 0.55


def _torch_slice(q1, k1, q2, k2, g, scale, causal):
    """KL, lse1, lse2 rows and the four gradients of sum_i g_i KL_i for one
    (b, h) slice, by torch fp64 autograd over sliced (not masked) rows."""
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q1, k1, q2, k2)]
    n_q, n_k = q1.shape[0], k1.shape[0]
    kls = []
    for i in range(n_q):
        n = n_k if not causal else i + 1 + (n_k - n_q)
        lp1 = torch.log_softmax(scale * t[1][:n] @ t[0][i], dim=-1)
        lp2 = torch.log_softmax(scale * t[3][:n] @ t[2][i], dim=-1)
        kls.append(torch.nn.functional.kl_div(lp2, lp1, reduction="sum", log_target=True))
    kl = torch.stack(kls)
    (kl * torch.tensor(g)).sum().backward()
    # order of the oracle's outputs: dq2, dk2, dq1, dk1
    return kl.detach().numpy(), [t[2].grad.numpy(), t[3].grad.numpy(), t[0].grad.numpy(),
                                 t[1].grad.numpy()]


@pytest.mark.parametrize("causal", [False, True])
def test_batched_forward_and_backward_per_slice(causal):
    """The batched [B, H] entry points against routes that share nothing with
    the oracle: scipy row loops for KL and LSE, torch fp64 autograd for the
    four gradients, slice by slice."""
    q1, k1, q2, k2, g, scale = _batched_case()
    B, H, n_q, _ = q1.shape
    n_k = k1.shape[2]
    kl, lse1, lse2 = orc.forward(q1, k1, q2, k2, scale, causal)
    grads = orc.backward(q1, k1, q2, k2, scale, causal, g, True)
    assert kl.shape == lse1.shape == lse2.shape == (B, H, n_q)
    assert grads[0].shape == grads[2].shape == q1.shape
    assert grads[1].shape == grads[3].shape == k1.shape
    for b in range(B):
        for h in range(H):
            for i in range(n_q):
                n = n_k if not causal else i + 1 + (n_k - n_q)
                s1 = scale * (k1[b, h, :n] @ q1[b, h, i])
                s2 = scale * (k2[b, h, :n] @ q2[b, h, i])
                assert kl[b, h, i] == pytest.approx(
                    sst.entropy(sps.softmax(s1), sps.softmax(s2)), rel=1e-10, abs=1e-13)
                assert lse1[b, h, i] == pytest.approx(sps.logsumexp(s1), rel=1e-13)
                assert lse2[b, h, i] == pytest.approx(sps.logsumexp(s2), rel=1e-13)
            _, ref = _torch_slice(q1[b, h], k1[b, h], q2[b, h], k2[b, h], g[b, h], scale, causal)
            for got, want in zip(grads, ref):
                np.testing.assert_allclose(got[b, h], want, rtol=1e-9, atol=1e-13)


def test_batched_one_gradient_set_and_head_subset():
    """grad1 = False returns only configuration 1's gradients; a head subset
    leaves the other heads NaN and is exact on its own heads."""
    q1, k1, q2, k2, g, scale = _batched_case()
    full = orc.backward(q1, k1, q2, k2, scale, True, g, True)
    one = orc.backward(q1, k1, q2, k2, scale, True, g, False)
    assert one[2] is None and one[3] is None
    np.testing.assert_array_equal(one[0], full[0])
    np.testing.assert_array_equal(one[1], full[1])
    sub = orc.backward(q1, k1, q2, k2, scale, True, g, True, heads=[(1, 2)])
    fsub = orc.forward(q1, k1, q2, k2, scale, True, heads=[(1, 2)])
    for x, y in zip(sub, full):
        np.testing.assert_array_equal(x[1, 2], y[1, 2])
        assert np.all(np.isnan(x[0])) and np.all(np.isnan(x[1, :2]))
    assert np.all(np.isnan(fsub[0][0])) and np.all(np.isfinite(fsub[0][1, 2]))


@pytest.mark.parametrize("mutation", ["q1_q2_k1_k2", "swap_student_teacher", "swap_lse_outputs",
                                      "g_other_head", "dq_dk_sets_swapped"])
def test_batched_planted_mistakes_are_caught(monkeypatch, mutation):
    """Plausible slips at the batched entry points' call sites (arguments or
    outputs in the wrong order, the wrong slice of g) fail the per-slice pin."""
    real_f, real_b = orc.head_forward, orc.head_backward
    if mutation == "q1_q2_k1_k2":  # N_Q != N_K: the shapes no longer line up
        monkeypatch.setattr(orc, "head_forward",
                            lambda q1, k1, q2, k2, *a, **k: real_f(q1, q2, k1, k2, *a, **k))
    elif mutation == "swap_student_teacher":
        monkeypatch.setattr(orc, "head_forward",
                            lambda q1, k1, q2, k2, *a, **k: real_f(q2, k2, q1, k1, *a, **k))
    elif mutation == "swap_lse_outputs":
        def f(*a, **k):
            kl, l1, l2 = real_f(*a, **k)
            return kl, l2, l1
        monkeypatch.setattr(orc, "head_forward", f)
    elif mutation == "g_other_head":
        def b(q1, k1, q2, k2, scale, causal, g, grad1, rows=None):
            return real_b(q1, k1, q2, k2, scale, causal, g[::-1].copy(), grad1, rows)
        monkeypatch.setattr(orc, "head_backward", b)
    else:
        def b(*a, **k):
            dq2, dk2, dq1, dk1 = real_b(*a, **k)
            return dq1, dk1, dq2, dk2
        monkeypatch.setattr(orc, "head_backward", b)
    with pytest.raises((AssertionError, ValueError)):
        test_batched_forward_and_backward_per_slice(True)


def test_backward_rejects_causal_with_more_queries_than_keys():
    q1, k1, q2, k2 = _case(43, 9, 5, 4)
    with pytest.raises(ValueError):
        orc.head_backward(q1, k1, q2, k2, 0.5, True, np.ones(9), True)
    with pytest.raises(ValueError):
        orc.head_forward(q1, k1, q2, k2, 0.5, True)
