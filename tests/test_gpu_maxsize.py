"""The largest sequence the C ABI accepts (N = 2^20 = 1048576), forward and backward, causal.

The oracle cannot materialise a 2^20 x 2^20 score matrix, so it checks what it can compute
exactly one piece at a time (tolerances of tests/parity.py):
* the first four query rows (they see keys 0..3 only) and one middle row: O, L, dQ;
* the last five query rows against all keys: O, L, dQ, and dK, dV of the last five keys,
  which no earlier query sees;
and two identities that hold at any size: sum_j dV_j = sum_i dO_i (every row of P sums to
1) and sum_j dK_j = 0 (every row of dS = P * (dP - D) sums to 0).
"""
import numpy as np
import pytest
import torch

import oracle.attention as OA
from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

from parity import GRAD_TOL, LSE_TOL, o_error, rel_fro

pytestmark = pytest.mark.gpu

N = 1 << 20


def _f64(x):
    return x.detach().cpu().double().numpy()


def test_maximum_length_sampled_rows_and_identities():
    w = I.custom(1, 1, N, 128, "bf16", True, seed=77)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    for t in (o, lse, dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    Q, K, V, DO = (_f64(x[0, 0]) for x in (q, k, v, do))
    O, L, DQ, DK, DV = (_f64(x[0, 0]) for x in (o, lse, dq, dk, dv))

    def check_rows(rows, ref):
        r = o_error(O[rows], ref["o"], w.torch_dtype)
        assert r["o_excess"] <= 0, (rows, r["o_max"])
        assert np.abs(L[rows] - ref["lse"]).max() <= LSE_TOL, rows
        assert rel_fro(DQ[rows], ref["dq"]) <= GRAD_TOL, rows

    # first rows: they see keys 0..3 only
    check_rows(slice(0, 4), OA.attention_backward(Q[:4], K[:4], V[:4], DO[:4], True, w.scale))
    # a middle row against its keys 0..i
    i = (N >> 1) + 7
    check_rows(slice(i, i + 1), OA.attention_backward(Q[i:i + 1], K[:i + 1], V[:i + 1],
                                                      DO[i:i + 1], True, w.scale))
    # last rows against all keys (bottom-right alignment: query t sees keys <= N - 5 + t)
    ref = OA.attention_backward(Q[N - 5:], K, V, DO[N - 5:], True, w.scale)
    check_rows(slice(N - 5, N), ref)
    assert rel_fro(DK[N - 5:], ref["dk"][N - 5:]) <= GRAD_TOL
    assert rel_fro(DV[N - 5:], ref["dv"][N - 5:]) <= GRAD_TOL
    # identities over all keys
    sum_dv, sum_do = DV.sum(axis=0), DO.sum(axis=0)
    assert np.linalg.norm(sum_dv - sum_do) <= GRAD_TOL * np.linalg.norm(sum_do)
    # The exact sum is 0. What is left is the rounding of 2^20 independent rows: about
    # sqrt(N) * (16-bit rounding) * rms(dK_j), i.e. a small fraction of ||dK||_F.
    sum_dk = DK.sum(axis=0)
    assert np.linalg.norm(sum_dk) <= GRAD_TOL * np.linalg.norm(DK)
