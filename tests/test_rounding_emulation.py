"""Why the O bound allows half an output ulp on top of 1e-2 where |O_ref| >= 2.

The forward rounds the probabilities P to the input type before the product P V
("Triton 05: Flash Attention", section 코드 라인별 설명 (Forward), step 5: p.to(v.dtype))
and stores O in the input type. This CPU test emulates those roundings step by step on
the softmax-stress workload (B2 H32 N8192 d64 bf16, q and k x4, +8 on 1% of late keys)
and measures, against the fp64 oracle on the same inputs:

  * before storage (O = acc / l-hat kept in float64) the error stays below 1e-2 on every
    element: the computation itself meets the 1e-2 budget;
  * after O is rounded to bf16 the error stays below 1e-2 wherever |O_ref| < 2, but some
    elements with |O_ref| >= 2 exceed it, all of them by less than half an ulp of bf16
    (0.0078 in [2, 4)): storage rounding, which no kernel that writes bf16 can avoid.

The emulated kernel is the textbook tile recurrence with the roundings of the CUDA
kernels: scores in float32, exponentials in float32 (base 2, scale * log2(e) folded),
a running max that moves only when the block max exceeds it by more than 8 (log2
units), P rounded to bf16 for P V, the denominator summed over the same rounded values.
It uses the oracle only for the reference O. This file holds test arithmetic only; it
shares nothing with the CUDA path.
"""
import numpy as np
import pytest
import torch

import oracle.attention as OA
from exact_attention_tcgen05_gb300 import inputs as I

from parity import O_STORAGE_FROM, O_TOL, ulp

W = I.BY_NAME["B2_H32_N8192_d64_bf16_full_spiked"]
LOG2E = 1.4426950408889634


def _bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.bfloat16().float().numpy().astype(np.float64)


def _emulated_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                      block: int = 128, rescale_threshold: float = 8.0) -> np.ndarray:
    """O before storage rounding, as the tile recurrence with bf16 P computes it."""
    s_all = (q @ k.T).astype(np.float32) * np.float32(scale * LOG2E)
    n = q.shape[0]
    m = np.full(n, -np.inf, dtype=np.float32)
    l_hat = np.zeros(n)
    acc = np.zeros((n, v.shape[1]))
    for j0 in range(0, k.shape[0], block):
        s = s_all[:, j0:j0 + block]
        m_cand = s.max(axis=1)
        move = m_cand > m + np.float32(rescale_threshold)
        # (min(., 0) and the ignored -inf - -inf only touch rows where the max stays)
        with np.errstate(invalid="ignore"):
            alpha = np.where(move, np.exp2(np.minimum(m - m_cand, 0)), 1.0)
        m = np.where(move, m_cand, m)
        p = np.exp2(s - m[:, None], dtype=np.float32)
        p_hat = _bf16(p)
        l_hat = l_hat * alpha + p_hat.sum(axis=1)
        acc = acc * alpha[:, None] + p_hat @ v[j0:j0 + block]
    return acc / l_hat[:, None]


@pytest.mark.slow
def test_bf16_storage_not_computation_exceeds_flat_bound():
    before, after_small, over = 0.0, 0.0, []
    for b, h in I.sampled_slices(W):
        q, k, v = (I.to_f64(I.make_slice(W, b, h, t)) for t in ("q", "k", "v"))
        o_ref, _ = OA.attention_forward(q, k, v, W.causal, W.scale)
        for r0 in range(0, W.N, 2048):
            rows = slice(r0, r0 + 2048)
            pre = _emulated_forward(q[rows], k, v, W.scale)
            ref = o_ref[rows]
            stored = _bf16(pre)
            err_pre = np.abs(pre - ref)
            err = np.abs(stored - ref)
            big = np.abs(ref) >= O_STORAGE_FROM
            before = max(before, float(err_pre.max()))
            after_small = max(after_small, float(err[~big].max()))
            sel = big & (err > O_TOL)
            over += list(zip(err[sel], ref[sel]))
    # the computation meets the budget on every element
    assert before <= O_TOL, before
    # stored bf16 values still do where half an ulp is at most 0.0039
    assert after_small <= O_TOL, after_small
    # ... but not everywhere: some stored values with |O_ref| >= 2 exceed 1e-2, each by
    # less than the half ulp the bound allows there
    assert over, "expected elements with |O_ref| >= 2 above 1e-2 after bf16 storage"
    for e, r in over:
        assert e <= O_TOL + 0.5 * float(ulp(np.array([r]), torch.bfloat16)[0]), (e, r)


def test_emulation_is_the_oracle_without_roundings():
    """With no rounding (fp64 scores, exponentials and P) and every block rescaled, the
    emulated recurrence reproduces the oracle to fp64 accuracy: the emulation above
    differs from the definition only in the roundings it adds."""
    w = I.custom(1, 1, 300, 64, "bf16", False, seed=9, qk_gain=4.0)
    q, k, v = (I.to_f64(I.make_slice(w, 0, 0, t)) for t in ("q", "k", "v"))
    o_ref, _ = OA.attention_forward(q, k, v, False, w.scale)
    s_all = (q @ k.T) * (w.scale * LOG2E)
    m = np.full(300, -np.inf)
    l = np.zeros(300)
    acc = np.zeros((300, 64))
    for j0 in range(0, 300, 128):
        s = s_all[:, j0:j0 + 128]
        m_new = np.maximum(m, s.max(axis=1))
        alpha = np.exp2(m - m_new)
        p = np.exp2(s - m_new[:, None])
        l = l * alpha + p.sum(axis=1)
        acc = acc * alpha[:, None] + p @ v[j0:j0 + 128]
        m = m_new
    assert np.abs(acc / l[:, None] - o_ref).max() < 1e-12
