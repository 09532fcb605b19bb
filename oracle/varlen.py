"""fp64 CPU oracle for attention over variable-length sequences packed along the token axis.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this module.

Source: "FlashAttentionを1から — 計算を増やして速くする逆説", section 現場ではこう使う,
the last pitfall: a batch of sentences of different lengths padded to the longest one
pays for the padded positions in both computation and memory traffic; the
variable-length interface, which takes the sequence boundaries as ``cu_seqlens``, does
not (the same section names ``flash_attn_varlen_func``).

Reading (the page names the interface but not its layout; this is the plainest layout
that matches it):

* B sequences lie one after another along the token axis. q, o, dO, dq are
  [total_q, H, d]; k, v, dk, dv are [total_k, H, d]; lse and D are [H, total_q].
* ``cu_q`` and ``cu_k`` are the B + 1 cumulative lengths (cu[0] = 0, non-decreasing,
  cu[B] = total): sequence b owns query tokens cu_q[b] .. cu_q[b+1] - 1 and key tokens
  cu_k[b] .. cu_k[b+1] - 1.
* Each (sequence, head) pair is an independent attention problem, exactly the one of
  ``oracle.attention`` on that sequence's rows: its queries see only its own keys, with
  the causal mask bottom-right aligned within the sequence (key j of the sequence is
  visible to its query i iff j <= i + (n_k - n_q)). Tokens of other sequences take no
  part, so no padding is computed and nothing else is masked.

Every function here is pinned in tests/test_varlen_oracle.py (brute force, the pages'
worked example placed among other sequences, isolation of sequences, finite
differences).
"""
from __future__ import annotations

import numpy as np

import oracle.attention as OA


def _bounds(cu: np.ndarray, b: int) -> tuple[int, int]:
    return int(cu[b]), int(cu[b + 1])


def _check_pair(nq: int, nk: int, causal: bool) -> None:
    # A sequence with queries must have a key every query sees: at least one key, and
    # with the mask at least as many keys as queries (else its first rows see nothing).
    if nq > 0 and (nk == 0 or (causal and nk < nq)):
        raise ValueError("a sequence has queries that see no key")


def check_cu(cu, total: int) -> np.ndarray:
    """cu_seqlens as an int array; raises on a malformed one."""
    cu = np.asarray(cu, dtype=np.int64)
    if (cu.ndim != 1 or cu.size < 2 or cu[0] != 0 or cu[-1] != total
            or np.any(np.diff(cu) < 0)):
        raise ValueError("cu_seqlens must start at 0, not decrease and end at the total")
    return cu


def varlen_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_q, cu_k, causal: bool,
                   scale: float) -> tuple[np.ndarray, np.ndarray]:
    """O [total_q, H, d] and L [H, total_q] (natural log) of every packed sequence."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    cu_q, cu_k = check_cu(cu_q, q.shape[0]), check_cu(cu_k, k.shape[0])
    H = q.shape[1]
    o = np.zeros((q.shape[0], H, v.shape[2]))
    lse = np.zeros((H, q.shape[0]))
    for b in range(cu_q.size - 1):
        q0, q1 = _bounds(cu_q, b)
        k0, k1 = _bounds(cu_k, b)
        _check_pair(q1 - q0, k1 - k0, causal)
        if q1 == q0:
            continue
        for h in range(H):
            ob, lb = OA.attention_forward(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], causal, scale)
            o[q0:q1, h] = ob
            lse[h, q0:q1] = lb
    return o, lse


def varlen_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, do: np.ndarray, cu_q, cu_k,
                    causal: bool, scale: float) -> dict:
    """dq [total_q, H, d], dk and dv [total_k, H, d] of sum(dO * O), with the forward's o,
    lse and D = rowsum(dO * O) ([H, total_q])."""
    q, k, v, do = (np.asarray(x, dtype=np.float64) for x in (q, k, v, do))
    cu_q, cu_k = check_cu(cu_q, q.shape[0]), check_cu(cu_k, k.shape[0])
    H = q.shape[1]
    out = dict(dq=np.zeros_like(q), dk=np.zeros_like(k), dv=np.zeros_like(v),
               o=np.zeros((q.shape[0], H, v.shape[2])), lse=np.zeros((H, q.shape[0])),
               delta=np.zeros((H, q.shape[0])))
    for b in range(cu_q.size - 1):
        q0, q1 = _bounds(cu_q, b)
        k0, k1 = _bounds(cu_k, b)
        _check_pair(q1 - q0, k1 - k0, causal)
        if q1 == q0:
            continue  # keys that no query sees get zero gradients
        for h in range(H):
            r = OA.attention_backward(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h],
                                      causal, scale)
            out["dq"][q0:q1, h] = r["dq"]
            out["dk"][k0:k1, h] = r["dk"]
            out["dv"][k0:k1, h] = r["dv"]
            out["o"][q0:q1, h] = r["o"]
            out["lse"][h, q0:q1] = r["lse"]
            out["delta"][h, q0:q1] = r["delta_rowsum"]
    return out
