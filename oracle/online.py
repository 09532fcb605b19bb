"""The blocked online-softmax recurrence, written out step by step in fp64.

TEST INFRASTRUCTURE ONLY (same rule as ``oracle.attention``): it exists to check the
definition-based oracle against a second, independent statement of the method, and
to replay the pages' worked examples. Nothing on the product path calls it.

The state kept per query row, and its update when a new block of keys arrives, follow
"FlashAttention·FA4·FP4 — Tri Dao 외, Ted Zadouri 외, Robert Hu의 최적화 연구"
(yousangson.github.io), section 온라인 softmax가 블록 사이의 값을 어떻게 이어 주나
(how online softmax joins blocks), in that page's notation:

* m: the largest score seen so far;
* l: the sum of exp(s_j - m) over the keys seen so far;
* u: the matching unnormalised output, sum of exp(s_j - m) v_j.

For a new block with scores s_j and values v_j:
  m' = max(m, max_j s_j);  l' = exp(m - m') l + sum_j exp(s_j - m');
  u' = exp(m - m') u + sum_j exp(s_j - m') v_j.
After the last block the output is u / l (one final divide, as in "Triton 05: Flash
Attention", section 최종 정규화). The state starts at m = -inf, l = 0, u = 0, so the
first rescale factor exp(-inf) is 0 ("GPU에서 Attention은 실제로 어떻게 실행되는가",
Part 3-2 Online Softmax). The same three equations merge partial states computed
over disjoint key ranges ("FlashAttentionを1から", section その後の版と、推論での事情).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterable, Sequence

import numpy as np


@dataclasses.dataclass
class RowState:
    """Running statistics of one query row."""

    m: float
    l: float
    u: np.ndarray

    @staticmethod
    def empty(dv: int) -> "RowState":
        return RowState(-math.inf, 0.0, np.zeros(dv))


def rescale_factor(m_old: float, m_new: float) -> float:
    """exp(m_old - m_new); 0 when nothing was seen yet (m_old = -inf)."""
    if m_old == -math.inf:
        return 0.0
    return math.exp(m_old - m_new)


def absorb_block(state: RowState, s_block: np.ndarray, v_block: np.ndarray,
                 rescale: bool = True) -> RowState:
    """Fold one key block (scores s_block [n], values v_block [n, dv]) into the state.

    ``rescale=False`` drops the exp(m - m') factor; it exists only so that a test can
    show that the pages' negative control (which omits it) gives a different answer.
    """
    s_block = np.asarray(s_block, dtype=np.float64)
    v_block = np.asarray(v_block, dtype=np.float64).reshape(len(s_block), -1)
    visible = s_block > -math.inf
    if not visible.any():
        return state
    m_new = max(state.m, float(s_block[visible].max()))
    alpha = rescale_factor(state.m, m_new) if rescale else (
        0.0 if state.m == -math.inf else 1.0)
    w = np.where(visible, np.exp(np.where(visible, s_block, 0.0) - m_new), 0.0)
    return RowState(m_new, alpha * state.l + float(w.sum()), alpha * state.u + w @ v_block)


def merge(a: RowState, b: RowState) -> RowState:
    """Combine two partial states over disjoint key ranges."""
    m_new = max(a.m, b.m)
    if m_new == -math.inf:
        return RowState(m_new, 0.0, np.zeros_like(a.u))
    fa, fb = rescale_factor(a.m, m_new), rescale_factor(b.m, m_new)
    return RowState(m_new, fa * a.l + fb * b.l, fa * a.u + fb * b.u)


def finish(state: RowState) -> tuple[np.ndarray, float]:
    """Output u / l and natural-log LSE m + ln l of a finished row."""
    return state.u / state.l, state.m + math.log(state.l)


def row_blocks(n: int, block: int) -> Iterable[tuple[int, int]]:
    for j0 in range(0, n, block):
        yield j0, min(n, j0 + block)


def run_row(s_row: Sequence[float], values: np.ndarray, block: int,
            rescale: bool = True) -> tuple[np.ndarray, float, list[RowState]]:
    """Stream one row of (already scaled, masked) scores through the recurrence.

    Returns the output, the LSE and the state after every block.
    """
    s_row = np.asarray(s_row, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64).reshape(len(s_row), -1)
    st = RowState.empty(values.shape[1])
    trace = []
    for j0, j1 in row_blocks(len(s_row), block):
        st = absorb_block(st, s_row[j0:j1], values[j0:j1], rescale)
        trace.append(dataclasses.replace(st, u=st.u.copy()))
    o, lse = finish(st)
    return o, lse, trace


def blocked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, causal: bool,
                      scale: float, block_q: int, block_k: int
                      ) -> tuple[np.ndarray, np.ndarray]:
    """The whole [N, d] slice by blocks: query blocks of block_q rows, each streaming
    key blocks of block_k keys. Score blocks are formed one at a time; no N x N array
    exists. Causal masking puts -inf on keys j > i inside each score block.
    """
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    n, dv = q.shape[0], v.shape[1]
    o = np.empty((n, dv))
    lse = np.empty(n)
    for i0, i1 in row_blocks(n, block_q):
        states = [RowState.empty(dv) for _ in range(i0, i1)]
        for j0, j1 in row_blocks(k.shape[0], block_k):
            if causal and j0 > i1 - 1:
                break
            s_blk = scale * (q[i0:i1] @ k[j0:j1].T)
            if causal:
                ii = np.arange(i0, i1)[:, None]
                jj = np.arange(j0, j1)[None, :]
                s_blk = np.where(jj > ii, -np.inf, s_blk)
            for r in range(i1 - i0):
                states[r] = absorb_block(states[r], s_blk[r], v[j0:j1])
        for r, st in enumerate(states):
            o[i0 + r], lse[i0 + r] = finish(st)
    return o, lse
