"""Head dims above 128 (136 to 256, multiples of 8): the 256-column forward and the three
passes of the 256-column backward (dQ; dV, then dK) against the fp64 oracle, element by
element, with the tolerances of tests/parity.py.

The cases span several 128-row tiles and 64-key blocks with ragged tails, one-row and
one-block sequences, head dims that leave zero-read columns in the 256-column tiles, N_q
against N_k with bottom-right causal masking, and a larger multi-head case compared on
sampled slices.
"""
import numpy as np
import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

from parity import GpuRun, all_finite, assert_within, compare_slice, record, run_gpu

pytestmark = pytest.mark.gpu

WIDE = [
    # (B, H, N, d, dtype, causal)
    (1, 2, 256, 256, "bf16", False),
    (1, 2, 300, 256, "fp16", True),
    (2, 1, 513, 256, "bf16", True),
    (1, 1, 1000, 192, "bf16", True),
    (1, 2, 129, 136, "fp16", False),
    (1, 1, 700, 248, "bf16", False),
    (1, 2, 65, 256, "bf16", True),
    (1, 1, 2048, 256, "fp16", False),  # 32 key blocks: the rescale path over a long row
]


@pytest.mark.parametrize("shape", WIDE, ids=lambda s: "B{}H{}N{}d{}_{}_{}".format(
    *s[:5], "causal" if s[5] else "full"))
def test_wide_all_slices(shape):
    B, H, N, d, dt, causal = shape
    w = I.custom(B, H, N, d, dt, causal, seed=11 + N + d)
    run = run_gpu(w)
    assert run.o.shape == (B, H, N, d) and run.dk.shape == (B, H, N, d)
    assert all_finite(run)
    assert binding.attn_last_kernel_status() == (0, 0)
    for b in range(B):
        for h in range(H):
            res = compare_slice(w, run, b, h)
            record(f"wide {w.name}", res)
            assert_within(res, f"{w.name} slice {(b, h)}")


@pytest.mark.parametrize("Nq,Nk,d,causal", [(300, 777, 256, True), (1, 1000, 192, True),
                                            (200, 129, 256, False), (64, 129, 256, True),
                                            (128, 640, 256, True)])
def test_wide_rectangular(Nq, Nk, d, causal):
    wq = I.custom(1, 2, Nq, d, "bf16", causal, seed=50 + Nq)
    wk = I.custom(1, 2, Nk, d, "bf16", causal, seed=51 + Nk)
    q, do = (I.make_tensor(wq, t).cuda() for t in ("q", "do"))
    k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=wq.scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=wq.scale)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    run = GpuRun(q, k, v, do, o, lse, dq, dk, dv)
    assert dk.shape == (1, 2, Nk, d)
    assert all_finite(run)
    for h in range(2):
        assert_within(compare_slice(wq, run, 0, h), f"Nq{Nq} Nk{Nk} head {h}")


def test_wide_many_heads_sampled():
    w = I.custom(2, 8, 4096, 256, "bf16", True, seed=77)
    run = run_gpu(w)
    assert all_finite(run)
    assert binding.attn_last_kernel_status() == (0, 0)
    for b, h in [(0, 0), (1, 7), (0, 5)]:
        res = compare_slice(w, run, b, h)
        record(w.name, res)
        assert_within(res, f"{w.name} slice {(b, h)}")


@pytest.mark.parametrize("d,dt", [(256, "fp16"), (256, "bf16"), (200, "bf16")])
def test_wide_single_key_gradients_vanish(d, dt):
    """N = 1: P = 1, so dS = dP - D and dQ = dK = 0 exactly. The kernels form dP on the
    tensor core and D in the preprocess, two fp32 sums of the same d products in different
    orders; each is within 2 d u sum_c |dO_c V_c| of the exact dot (u = 2^-24, doubled for
    the tensor core's accumulation), so |dQ_c| <= scale |dS| |K_c| and |dK_c| <= scale |dS|
    |Q_c| with |dS| <= 4 d u sum_c |dO_c V_c| (times 1 + 2^-7 for the 16-bit roundings).
    O, L and dV = dO are compared with the oracle as everywhere else."""
    w = I.custom(1, 2, 1, d, dt, False, seed=268 + d)
    run = run_gpu(w)
    assert all_finite(run)
    for h in range(2):
        res = compare_slice(w, run, 0, h)
        assert res["o_excess"] <= 0.0 and res["lse_max"] <= 1e-3 and res["dv"] <= 3e-2
        q, k, v, do = (I.to_f64(x[0, h]) for x in (run.q, run.k, run.v, run.do))
        ds_max = 4 * d * 2.0 ** -24 * float(np.abs(do[0] * v[0]).sum()) * (1 + 2.0 ** -7)
        dq, dk = I.to_f64(run.dq[0, h]), I.to_f64(run.dk[0, h])
        assert np.all(np.abs(dq) <= w.scale * ds_max * np.abs(k) * (1 + 2.0 ** -7) + 1e-30)
        assert np.all(np.abs(dk) <= w.scale * ds_max * np.abs(q) * (1 + 2.0 ** -7) + 1e-30)


def test_head_dim_workload_sampled():
    """The head-dim-256 workload the benchmark times, at full size, on sampled slices."""
    w = I.BY_NAME["B4_H16_N4096_d256_bf16_causal"]
    run = run_gpu(w)
    assert all_finite(run)
    assert binding.attn_last_kernel_status() == (0, 0)
    for b, h in I.sampled_slices(w):
        res = compare_slice(w, run, b, h)
        record(w.name, res)
        assert_within(res, f"{w.name} slice {(b, h)}")
