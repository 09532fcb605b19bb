"""Head dims above 128 (136 to 256, multiples of 8): the 256-column forward against the fp64
oracle, element by element, with the tolerances of tests/parity.py.

The cases span several 128-row tiles and 64-key blocks with ragged tails, one-row and
one-block sequences, head dims that leave zero-read columns in the 256-column tiles, N_q
against N_k with bottom-right causal masking, and a larger multi-head case compared on
sampled slices.
"""
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
    (1, 1, 1, 256, "fp16", False),
    (1, 1, 2048, 256, "fp16", False),  # 32 key blocks: the rescale path over a long row
]


@pytest.mark.parametrize("shape", WIDE, ids=lambda s: "B{}H{}N{}d{}_{}_{}".format(
    *s[:5], "causal" if s[5] else "full"))
def test_wide_forward_all_slices(shape):
    B, H, N, d, dt, causal = shape
    w = I.custom(B, H, N, d, dt, causal, seed=11 + N + d)
    run = run_gpu(w, backward=False)
    assert run.o.shape == (B, H, N, d)
    assert all_finite(run)
    assert binding.attn_last_kernel_status() == (0, 0)
    for b in range(B):
        for h in range(H):
            res = compare_slice(w, run, b, h, backward=False)
            record(f"wide {w.name}", res)
            assert_within(res, f"{w.name} slice {(b, h)}")


@pytest.mark.parametrize("Nq,Nk,d,causal", [(300, 777, 256, True), (1, 1000, 192, True),
                                            (200, 129, 256, False), (64, 129, 256, True)])
def test_wide_forward_rectangular(Nq, Nk, d, causal):
    wq = I.custom(1, 2, Nq, d, "bf16", causal, seed=50 + Nq)
    wk = I.custom(1, 2, Nk, d, "bf16", causal, seed=51 + Nk)
    q = I.make_tensor(wq, "q").cuda()
    k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=wq.scale)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    run = GpuRun(q, k, v, torch.zeros_like(q), o, lse, None, None, None)
    assert all_finite(run)
    for h in range(2):
        assert_within(compare_slice(wq, run, 0, h, backward=False), f"Nq{Nq} Nk{Nk} head {h}")


def test_wide_forward_many_heads_sampled():
    w = I.custom(2, 8, 4096, 256, "bf16", True, seed=77)
    run = run_gpu(w, backward=False)
    assert all_finite(run)
    for b, h in [(0, 0), (1, 7), (0, 5)]:
        res = compare_slice(w, run, b, h, backward=False)
        record(w.name, res)
        assert_within(res, f"{w.name} slice {(b, h)}")


def test_wide_backward_is_unsupported():
    w = I.custom(1, 1, 128, 256, "bf16", True, seed=5)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    with pytest.raises(binding.AttnError) as e:
        binding.attn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    assert e.value.code == 2  # ATTN_ERR_UNSUPPORTED
