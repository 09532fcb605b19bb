"""fp64 CPU oracle for split-KV decoding: one query row per (b, h) against a long K/V.

TEST INFRASTRUCTURE ONLY (same rule as ``oracle.attention``): only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may import it.

The method, from "FlashAttentionを1から — 計算を増やして速くする逆説":

* section その後の版と、推論での事情: while generating, the query is a single token, so
  parallelising over query rows leaves the GPU idle; instead the K/V side is split, the
  partial results are computed in parallel, and they are joined with the three update
  equations of the online softmax, which gives the same answer as no split;
* section オンラインsoftmax: 途中経過を、後から縮める: each part carries m (its largest
  score), l (the sum of exp(s_j - m)) and O~ (the matching unnormalised weighted sum of
  value rows). Joining a part (m~, l~, O~_part) into a running state (m, l, O~):
      m' = max(m, m~)
      l' = e^(m - m') l + e^(m~ - m') l~
      O~' = e^(m - m') O~ + e^(m~ - m') O~_part
  and after the last part O = O~ / l once. The exported logsumexp is L = m + ln l
  (natural log, scores already scaled), as for the forward.

The split of the keys is part of the interface (the same rule is stated in
include/attn.h): with S splits of a sequence of Nk keys, every split spans
C = 64 * ceil(ceil(Nk / S) / 64) keys, split s covering [s C, min((s + 1) C, Nk)); a
split past the end is empty and contributes the neutral state (m = -inf, l = 0, O~ = 0).

Each function below is pinned in tests/test_decode_oracle.py: the merged result against
the plain definition (``oracle.attention.attention_forward``) for every split, the pages'
worked example, order independence, and neutral empty parts.
"""
from __future__ import annotations

import math

import numpy as np

SPLIT_ALIGN = 64  # keys; split lengths are multiples of this


def split_length(nk: int, num_splits: int) -> int:
    """C, the number of keys in every split but possibly the last ones."""
    per = -(-nk // num_splits)
    return SPLIT_ALIGN * (-(-per // SPLIT_ALIGN))


def split_bounds(nk: int, num_splits: int) -> list[tuple[int, int]]:
    """[k0, k1) of each split; empty splits have k0 == k1."""
    c = split_length(nk, num_splits)
    return [(min(nk, s * c), min(nk, (s + 1) * c)) for s in range(num_splits)]


def partial_state(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  k0: int, k1: int) -> tuple[float, float, np.ndarray]:
    """(m, l, O~) of keys [k0, k1) for one query row, from the definition:
    s_j = scale q.k_j, m = max_j s_j, l = sum_j exp(s_j - m), O~ = sum_j exp(s_j - m) v_j.
    An empty range gives the neutral state (-inf, 0, 0)."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    if k1 <= k0:
        return -math.inf, 0.0, np.zeros(v.shape[1])
    s = scale * (k[k0:k1] @ q)
    m = float(s.max())
    e = np.exp(s - m)
    return m, float(e.sum()), e @ v[k0:k1]


def merge_states(parts) -> tuple[float, float, np.ndarray]:
    """Joins partial states left to right with the three update equations."""
    m, l, u = -math.inf, 0.0, None
    for m_p, l_p, u_p in parts:
        u_p = np.asarray(u_p, dtype=np.float64)
        if u is None:
            u = np.zeros_like(u_p)
        m_new = max(m, m_p)
        if m_new == -math.inf:  # both neutral so far
            continue
        a = math.exp(m - m_new)      # 0 when m = -inf
        b = math.exp(m_p - m_new)    # 0 when the part is empty
        l = a * l + b * l_p
        u = a * u + b * u_p
        m = m_new
    return m, l, u


def finish(m: float, l: float, u: np.ndarray) -> tuple[np.ndarray, float]:
    """O = O~ / l and L = m + ln l."""
    return u / l, m + math.log(l)


def decode(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, num_splits: int
           ) -> tuple[np.ndarray, float, list]:
    """Split-KV decode of one query row q [d] against k, v [Nk, d]: the partial state of
    every split, then their merge. Returns (O [d], L, parts)."""
    parts = [partial_state(q, k, v, scale, k0, k1)
             for k0, k1 in split_bounds(k.shape[0], num_splits)]
    o, lse = finish(*merge_states(parts))
    return o, lse, parts
