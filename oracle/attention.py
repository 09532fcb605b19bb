"""fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this module.
The product path never calls it: it has no CPU fallback.

What it computes is the plain definition that the tiled method reaches exactly (up to
rounding order). Sources:

* "Triton 05: Flash Attention" (wonbeomjang.kr), sections 핵심 개념 / Attention 수식
  and Standard Attention의 문제: S = QK^T / sqrt(d), row softmax, O = PV, with
  ``sm_scale = d ** -0.5`` from its torch.autograd.Function wrapper.
* "FlashAttentionを1から — 計算を増やして速くする逆説", section タイリングを阻む、
  softmaxという壁: the safe softmax e^{s_j - m} / sum_k e^{s_k - m}, m = max_k s_k.
* "Triton 05: Flash Attention", section Causal Masking: future keys (j > i) are
  blocked before the softmax.
* "Triton 05: Flash Attention", sections LSE로 P 재계산 and Softmax Gradient: the
  forward keeps the per-row logsumexp L; the backward uses
  D_i = rowsum(dO_i * O_i) and the softmax gradient dS = P * (dP - D).

Readings where the pages are silent or garbled (the formulas of the LSE and of the
gradient were lost from the extracted text):

* L_i = m_i + ln(sum_j exp(S_ij - m_i)) in the natural log, with S already scaled.
* The gradients are the exact derivatives of the definition above:
  dV = P^T dO, dP = dO V^T, D_i = sum_j P_ij dP_ij, dS = P * (dP - D),
  dQ = scale * dS K, dK = scale * dS^T Q. D_i equals rowsum(dO_i * O_i) in exact
  arithmetic; both are computed and returned.
* Causal masking is bottom-right aligned: with N_q query rows and N_k >= N_q keys, key j
  is visible to query i iff j <= i + (N_k - N_q), i.e. the queries are the last N_q
  positions of the sequence (for N_q = N_k: j <= i). Every row sees at least key 0 and no
  row is fully masked. The pages only say that future tokens are blocked ("Triton 05",
  Causal Masking); placing the queries last is the reading for a query chunk that
  follows the keys already in the cache.

Rows are processed in panels of whole rows only to bound memory (S and P of one
N = 16384 head are 2 GiB each in fp64). Each row's softmax and output depend on that
row alone, so the panel size changes no forward value; in the backward it only
changes the order in which the per-row terms of dK and dV are summed.

Parity pins: every function here is pinned by tests/test_oracle_pins.py against the
pages' worked examples, closed forms, brute force and finite differences.
"""
from __future__ import annotations

import numpy as np

DEFAULT_PANEL_ELEMS = 1 << 24  # rows per panel = this // N (16 M doubles = 128 MiB)


def _panel_rows(n: int, panel_elems: int) -> int:
    return max(1, min(n, panel_elems // max(1, n)))


def scores(q: np.ndarray, k: np.ndarray, scale: float, causal: bool,
           row0: int = 0, row1: int | None = None) -> np.ndarray:
    """Scaled, masked scores S[row0:row1, :] = scale * Q K^T with -inf on
    j > i + (N_k - N_q) (bottom-right aligned; j > i when N_q = N_k)."""
    row1 = q.shape[0] if row1 is None else row1
    s = scale * (q[row0:row1] @ k.T)
    if causal:
        offset = k.shape[0] - q.shape[0]
        rows = np.arange(row0, row1)[:, None]
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > rows + offset, -np.inf, s)
    return s


def softmax_rows(s: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Safe softmax of each row. Returns (P, m, l) with m the row max and
    l = sum_j exp(s_j - m)."""
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m, l


def attention_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                      scale: float, panel_elems: int = DEFAULT_PANEL_ELEMS
                      ) -> tuple[np.ndarray, np.ndarray]:
    """O = softmax(scale * Q K^T [masked]) V and L = m + ln l, for one (b, h) slice.

    q: [N_q, d], k, v: [N_k, d] float64 (N_k >= N_q when causal). Returns O [N_q, d]
    and L [N_q] (natural log), float64.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, dv = q.shape[0], v.shape[1]
    o = np.empty((n, dv))
    lse = np.empty(n)
    step = _panel_rows(n, panel_elems)
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        p, m, l = softmax_rows(scores(q, k, scale, causal, r0, r1))
        o[r0:r1] = p @ v
        lse[r0:r1] = m + np.log(l)
    return o, lse


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray,
                       causal: bool, scale: float,
                       panel_elems: int = DEFAULT_PANEL_ELEMS) -> dict:
    """Gradients of sum(dO * O) with respect to Q, K, V, for one (b, h) slice.

    Returns a dict with dq, dk, dv [N, d], the two forms of D [N]
    (``delta`` = sum_j P_ij dP_ij and ``delta_rowsum`` = rowsum(dO * O)),
    and the forward outputs o, lse.
    """
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    n, d = q.shape
    dq = np.empty((n, d))
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.empty((n, v.shape[1]))
    lse = np.empty(n)
    delta = np.empty(n)
    delta_rowsum = np.empty(n)
    step = _panel_rows(n, panel_elems)
    for r0 in range(0, n, step):
        r1 = min(n, r0 + step)
        p, m, l = softmax_rows(scores(q, k, scale, causal, r0, r1))
        o_p = p @ v
        o[r0:r1] = o_p
        lse[r0:r1] = m + np.log(l)
        do_p = do[r0:r1]
        dv += p.T @ do_p
        dp = do_p @ v.T
        dlt = (p * dp).sum(axis=1)
        delta[r0:r1] = dlt
        delta_rowsum[r0:r1] = (do_p * o_p).sum(axis=1)
        ds = p * (dp - dlt[:, None])
        dq[r0:r1] = scale * (ds @ k)
        dk += scale * (ds.T @ q[r0:r1])
    return dict(dq=dq, dk=dk, dv=dv, delta=delta, delta_rowsum=delta_rowsum, o=o, lse=lse)


def delta_rowsum(o: np.ndarray, do: np.ndarray) -> np.ndarray:
    """D_i = sum_c dO_ic * O_ic (the backward's preprocess quantity)."""
    return (np.asarray(do, dtype=np.float64) * np.asarray(o, dtype=np.float64)).sum(axis=1)

