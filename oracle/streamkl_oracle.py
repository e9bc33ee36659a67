"""Plain fp64 CPU oracle for the attention-KL primitive (StreamKL).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this module. The product path (the
CUDA library and its Python binding) never calls it and shares no code with it.

What it computes, per batch b, head h and query row i, follows the pages titled
"StreamKL: Fast and Memory-Efficient KL Divergence for Boosting Attention
Distillation" (arXiv 2606.20005):

* Abstract (paperdance.org / fugumt.com): attention distillation minimises
  KL(P1 || P2) between a teacher attention distribution P1 and a student P2,
  P_t = softmax(S_t), S_t = scale * Q_t K_t^T (+ mask).
* gist.science technical summary, "Metodologia" section 1 (online formulation):
  the per-row objective L = acc/l1 + LSE2 - LSE1 with LSE_t = m_t + log l_t,
  kept as five running scalars (m1, m2, l1, l2, acc) while key tiles stream by.
* same summary, section 2 (recomputation strategy): only KL and LSE1/LSE2 are
  saved; P_t = exp(S_t - LSE_t) is regenerated for the backward pass, which has
  two configurations: (1) P1 fixed, gradients reach Q2, K2; (2) P2 fixed,
  gradients reach Q1, K1.
* same summary, section 3 ("Estabilidad Numerica"): the configuration-2 log
  ratio log(P1/P2) is formed from logit differences and the saved LSEs, never
  from logs of probabilities.

Everything here is the plain definition written out: each row is materialised
in fp64 (rows are grouped into blocks only so that numpy can vectorise; every
row's arithmetic is independent of the grouping), then

    lse_t[i] = M + log sum_j exp(s_t[i, j] - M),   M = max_j s_t[i, j]
    KL[i]    = sum_j p1[i, j] * ((s1[i, j] - lse1[i]) - (s2[i, j] - lse2[i]))

over the allowed keys j only. Masking (a reading, the pages only say "causal"):
key j is allowed for query i iff j <= i + (N_K - N_Q) (bottom-right aligned;
j <= i when N_Q == N_K). Masked keys are excluded, not given -inf.

Gradients of the loss L = sum_i g[i] * KL[i] use the explicit softmax Jacobian:

    dKL[i]/ds2[i, j] = p2[i, j] - p1[i, j]
    dKL[i]/ds1[i, j] = p1[i, j] * (log(p1/p2)[i, j] - KL[i])
    dQ_t = scale * dS_t @ K_t,   dK_t = scale * dS_t^T @ Q_t,   dS_t = g * dKL/ds_t

``head_forward_online`` restates the pages' five-scalar streaming update in
fp64 with arbitrary key-tile sizes; the tests pin the two forms against each
other and against closed forms, library routines and finite differences.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "allowed_count",
    "head_forward",
    "head_forward_online",
    "head_backward",
    "forward",
    "backward",
    "dkl_ds1",
    "dkl_ds2",
]

# Rows per numpy block. Only a vectorisation width: no row depends on another.
_ROW_BLOCK = 256


def allowed_count(i, n_q: int, n_k: int, causal: bool):
    """Number of keys query row ``i`` may attend (keys 0 .. count-1).

    Causal masks are bottom-right aligned: key j is allowed iff
    j <= i + (n_k - n_q). Works elementwise on integer arrays.
    """
    i = np.asarray(i)
    if not causal:
        return np.full(i.shape, n_k, dtype=np.int64)
    return np.minimum(n_k, i + 1 + (n_k - n_q)).astype(np.int64)


def _f64(x) -> np.ndarray:
    a = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(a)):
        raise ValueError("oracle inputs must be finite")
    return a


def _scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """S = scale * Q K^T for a block of query rows (fp64)."""
    return scale * (q @ k.T)


def _mask(rows: np.ndarray, n_q: int, n_k: int, causal: bool) -> np.ndarray:
    """Boolean [len(rows), n_k]: True where key j is allowed for query row."""
    cnt = allowed_count(rows, n_q, n_k, causal)
    return np.arange(n_k)[None, :] < cnt[:, None]


def _log_softmax_masked(s: np.ndarray, allowed: np.ndarray):
    """Row-wise log-sum-exp and log-probabilities over the allowed entries.

    Returns (lse [R], logp [R, n_k]); logp is 0 where the key is masked (its
    probability is excluded, the value is never used).
    """
    s_allowed = np.where(allowed, s, -np.inf)
    m = np.max(s_allowed, axis=1)
    e = np.where(allowed, np.exp(s - m[:, None]), 0.0)
    lse = m + np.log(np.sum(e, axis=1))
    logp = np.where(allowed, s - lse[:, None], 0.0)
    return lse, logp


def dkl_ds2(p1: np.ndarray, p2: np.ndarray) -> np.ndarray:
    """dKL/ds2 = p2 - p1 (configuration 1: teacher P1 held fixed)."""
    return p2 - p1


def dkl_ds1(p1: np.ndarray, log_ratio: np.ndarray, kl: np.ndarray) -> np.ndarray:
    """dKL/ds1 = p1 * (log(p1/p2) - KL) (configuration 2: student P2 fixed).

    ``log_ratio`` is (s1 - lse1) - (s2 - lse2), built from logits and the
    log-sum-exps, as the numerical-stability paragraph of the pages asks.
    """
    return p1 * (log_ratio - kl[:, None])


def head_forward(q1, k1, q2, k2, scale: float, causal: bool, rows=None):
    """KL, lse1, lse2 for one (batch, head) slice.

    q1, q2: [N_Q, d]; k1, k2: [N_K, d]. ``rows`` selects query rows (default:
    all). Returns three fp64 arrays of len(rows).
    """
    q1, k1, q2, k2 = (_f64(x) for x in (q1, k1, q2, k2))
    n_q, n_k = q1.shape[0], k1.shape[0]
    if causal and n_q > n_k:
        raise ValueError("causal needs N_Q <= N_K (bottom-right alignment)")
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    kl = np.empty(len(rows))
    lse1 = np.empty(len(rows))
    lse2 = np.empty(len(rows))
    for b0 in range(0, len(rows), _ROW_BLOCK):
        r = rows[b0:b0 + _ROW_BLOCK]
        hi = int(allowed_count(r.max(), n_q, n_k, causal))  # keys past hi are masked for all r
        allowed = _mask(r, n_q, n_k, causal)[:, :hi]
        s1 = _scores(q1[r], k1[:hi], scale)
        s2 = _scores(q2[r], k2[:hi], scale)
        l1, logp1 = _log_softmax_masked(s1, allowed)
        l2, logp2 = _log_softmax_masked(s2, allowed)
        p1 = np.where(allowed, np.exp(logp1), 0.0)
        kl[b0:b0 + len(r)] = np.sum(p1 * (logp1 - logp2), axis=1)
        lse1[b0:b0 + len(r)] = l1
        lse2[b0:b0 + len(r)] = l2
    return kl, lse1, lse2


def head_forward_online(q1, k1, q2, k2, scale: float, causal: bool, tile_sizes):
    """The pages' one-pass form: five running scalars per row, fp64.

    Keys are visited in consecutive tiles whose sizes cycle through
    ``tile_sizes``. Per tile, for each row (vectorised over rows):

        m_t'  = max(m_t, max_j s_t)
        l_t   = exp(m_t - m_t') l_t + sum_j exp(s_t - m_t')
        acc   = exp(m_1 - m_1') acc + sum_j exp(s1 - m_1') (s1 - s2)

    and at the end LSE_t = m_t + log l_t, KL = acc/l1 + LSE2 - LSE1.
    Tiles entirely past a row's causal frontier contribute nothing (skipped).
    """
    q1, k1, q2, k2 = (_f64(x) for x in (q1, k1, q2, k2))
    n_q, n_k = q1.shape[0], k1.shape[0]
    rows = np.arange(n_q)
    cnt = allowed_count(rows, n_q, n_k, causal)
    m1 = np.full(n_q, -np.inf)
    m2 = np.full(n_q, -np.inf)
    l1 = np.zeros(n_q)
    l2 = np.zeros(n_q)
    acc = np.zeros(n_q)
    j0 = 0
    t = 0
    sizes = list(tile_sizes)
    while j0 < n_k:
        j1 = min(n_k, j0 + sizes[t % len(sizes)])
        t += 1
        live = cnt > j0  # rows with at least one allowed key in this tile
        if np.any(live):
            r = rows[live]
            allowed = np.arange(j0, j1)[None, :] < cnt[r][:, None]
            s1 = _scores(q1[r], k1[j0:j1], scale)
            s2 = _scores(q2[r], k2[j0:j1], scale)
            m1n = np.maximum(m1[r], np.max(np.where(allowed, s1, -np.inf), axis=1))
            m2n = np.maximum(m2[r], np.max(np.where(allowed, s2, -np.inf), axis=1))
            a1 = np.exp(m1[r] - m1n)  # exp(-inf) = 0 on a row's first tile
            a2 = np.exp(m2[r] - m2n)
            e1 = np.where(allowed, np.exp(s1 - m1n[:, None]), 0.0)
            e2 = np.where(allowed, np.exp(s2 - m2n[:, None]), 0.0)
            diff = np.where(allowed, s1 - s2, 0.0)
            l1[r] = a1 * l1[r] + e1.sum(axis=1)
            l2[r] = a2 * l2[r] + e2.sum(axis=1)
            acc[r] = a1 * acc[r] + (e1 * diff).sum(axis=1)
            m1[r] = m1n
            m2[r] = m2n
        j0 = j1
    lse1 = m1 + np.log(l1)
    lse2 = m2 + np.log(l2)
    kl = acc / l1 + lse2 - lse1
    return kl, lse1, lse2


def head_backward(q1, k1, q2, k2, scale: float, causal: bool, g, grad1: bool,
                  rows=None):
    """Gradients of L = sum_i g[i] KL[i] for one (batch, head) slice.

    Recomputes P1, P2 and KL itself from the inputs (it takes no saved state).
    ``rows`` restricts the sum over i to those query rows (default: all), so
    dK receives only their contributions and dQ is returned for them only.
    Returns (dq2, dk2, dq1, dk1); dq1/dk1 are None unless ``grad1``.
    """
    q1, k1, q2, k2 = (_f64(x) for x in (q1, k1, q2, k2))
    g = _f64(g)
    n_q, n_k = q1.shape[0], k1.shape[0]
    if causal and n_q > n_k:
        raise ValueError("causal needs N_Q <= N_K (bottom-right alignment)")
    rows = np.arange(n_q) if rows is None else np.asarray(rows, dtype=np.int64)
    dq2 = np.zeros((len(rows), q2.shape[1]))
    dk2 = np.zeros_like(k2)
    dq1 = np.zeros((len(rows), q1.shape[1])) if grad1 else None
    dk1 = np.zeros_like(k1) if grad1 else None
    for b0 in range(0, len(rows), _ROW_BLOCK):
        r = rows[b0:b0 + _ROW_BLOCK]
        hi = int(allowed_count(r.max(), n_q, n_k, causal))
        allowed = _mask(r, n_q, n_k, causal)[:, :hi]
        s1 = _scores(q1[r], k1[:hi], scale)
        s2 = _scores(q2[r], k2[:hi], scale)
        _, logp1 = _log_softmax_masked(s1, allowed)
        _, logp2 = _log_softmax_masked(s2, allowed)
        p1 = np.where(allowed, np.exp(logp1), 0.0)
        p2 = np.where(allowed, np.exp(logp2), 0.0)
        log_ratio = logp1 - logp2  # 0 on masked keys, where p1 = p2 = 0
        kl = np.sum(p1 * log_ratio, axis=1)
        gr = g[r][:, None]
        ds2 = gr * dkl_ds2(p1, p2)
        dq2[b0:b0 + len(r)] = scale * (ds2 @ k2[:hi])
        dk2[:hi] += scale * (ds2.T @ q2[r])
        if grad1:
            ds1 = gr * dkl_ds1(p1, log_ratio, kl)
            dq1[b0:b0 + len(r)] = scale * (ds1 @ k1[:hi])
            dk1[:hi] += scale * (ds1.T @ q1[r])
    return dq2, dk2, dq1, dk1


def forward(q1, k1, q2, k2, scale: float, causal: bool, heads=None):
    """Batched forward over [B, H, N, d] arrays.

    ``heads`` is an optional list of (b, h) pairs to compute (others are left
    NaN); heads are independent, so a subset is exact for those heads.
    Returns kl, lse1, lse2 as [B, H, N_Q] fp64.
    """
    q1 = np.asarray(q1)
    B, H, n_q, _ = q1.shape
    out = [np.full((B, H, n_q), np.nan) for _ in range(3)]
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in pairs:
        res = head_forward(q1[b, h], k1[b, h], q2[b, h], k2[b, h], scale, causal)
        for o, v in zip(out, res):
            o[b, h] = v
    return tuple(out)


def backward(q1, k1, q2, k2, scale: float, causal: bool, g, grad1: bool,
             heads=None):
    """Batched backward over [B, H, N, d] arrays; ``g`` is [B, H, N_Q].

    Returns (dq2, dk2, dq1, dk1) as fp64 arrays shaped like the inputs
    (dq1/dk1 None unless ``grad1``); heads outside ``heads`` are NaN.
    """
    q1 = np.asarray(q1)
    k1 = np.asarray(k1)
    outs = [np.full(q1.shape, np.nan), np.full(k1.shape, np.nan)]
    if grad1:
        outs += [np.full(q1.shape, np.nan), np.full(k1.shape, np.nan)]
    B, H = q1.shape[:2]
    pairs = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in pairs:
        res = head_backward(q1[b, h], k1[b, h], q2[b, h], k2[b, h], scale, causal,
                            np.asarray(g)[b, h], grad1)
        for o, v in zip(outs, res):
            o[b, h] = v
    if not grad1:
        outs += [None, None]
    return tuple(outs)
