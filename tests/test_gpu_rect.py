"""N_q query rows against N_k keys (attn_fwd_qk / attn_bwd_qk through the binding) versus
the fp64 oracle, element by element on every (b, h) slice, with the tolerances of
tests/parity.py.

Causal masking is bottom-right aligned: key j is visible to query i iff
j <= i + (N_k - N_q). The cases put the offset N_k - N_q on and off the 128-row and
64-key tile boundaries, make both lengths ragged, and include N_q = 1 (one query row
against a whole cache) and N_k < N_q without the mask.
"""
import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

from parity import GpuRun, all_finite, assert_within, compare_slice

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, dtype, causal
    (1, 2, 128, 512, 128, "bf16", True),     # offset a multiple of both tiles
    (1, 2, 300, 777, 64, "fp16", True),      # ragged both, offset 477
    (2, 1, 1, 1000, 128, "bf16", True),      # one query row: sees every key
    (1, 2, 64, 129, 128, "fp16", True),      # half a query tile, offset 65
    (1, 1, 513, 1100, 128, "bf16", True),    # five query tiles, offset 587
    (1, 2, 256, 4096, 64, "bf16", True),     # a chunk at the end of a long sequence
    (1, 2, 200, 333, 128, "bf16", False),
    (2, 1, 1000, 130, 64, "fp16", False),    # more queries than keys, no mask
    (1, 1, 17, 17, 128, "bf16", True),       # N_q = N_k: attn_fwd's own alignment
    (1, 2, 100, 333, 48, "fp16", True),      # a head dim of 48
]


def _run(B, H, Nq, Nk, d, dtype, causal, seed):
    wq = I.custom(B, H, Nq, d, dtype, causal, seed=seed)
    wk = I.custom(B, H, Nk, d, dtype, causal, seed=seed + 1)
    q, do = (I.make_tensor(wq, t).cuda() for t in ("q", "do"))
    k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=wq.scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=wq.scale)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    return wq, GpuRun(q, k, v, do, o, lse, dq, dk, dv)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}Nq{}Nk{}d{}_{}_{}".format(
    *c[:6], "causal" if c[6] else "full"))
def test_rectangular_all_slices(case):
    B, H, Nq, Nk, d, dtype, causal = case
    w, run = _run(*case, seed=40 + Nq + Nk)
    assert run.o.shape == (B, H, Nq, d) and run.lse.shape == (B, H, Nq)
    assert run.dq.shape == (B, H, Nq, d) and run.dk.shape == (B, H, Nk, d)
    assert all_finite(run)
    for b in range(B):
        for h in range(H):
            assert_within(compare_slice(w, run, b, h), f"{case} slice {(b, h)}")


def test_rectangular_many_items_sampled():
    """B4 H40, N_q = 640 against N_k = 1000: more work items than SMs in all three kernels,
    so they walk the host-computed greedy orders (item costs from the offset); sampled
    slices against the oracle."""
    case = (4, 40, 640, 1000, 64, "bf16", True)
    w, run = _run(*case, seed=2000)
    assert all_finite(run)
    for b, h in [(0, 0), (1, 17), (2, 31), (3, 39)]:
        assert_within(compare_slice(w, run, b, h), f"{case} slice {(b, h)}")


@pytest.mark.parametrize("Nq,Nk,d", [(192, 700, 128), (100, 355, 64)])
def test_keys_past_each_row_do_not_leak(Nq, Nk, d):
    """Changing keys j > i0 + (N_k - N_q) leaves rows i <= i0 of O and LSE bit-for-bit
    unchanged, and dK, dV of those keys are exactly zero when no later row sees them."""
    wq = I.custom(1, 2, Nq, d, "bf16", True, seed=9)
    wk = I.custom(1, 2, Nk, d, "bf16", True, seed=10)
    q, do = (I.make_tensor(wq, t).cuda() for t in ("q", "do"))
    k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
    off = Nk - Nq
    i0 = Nq // 2 + 3
    o, lse = binding.attn_fwd(q, k, v, causal=True, scale=wq.scale)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, i0 + off + 1:] *= -3
    v2[:, :, i0 + off + 1:] += 5
    o2, lse2 = binding.attn_fwd(q, k2, v2, causal=True, scale=wq.scale)
    torch.cuda.synchronize()
    assert torch.equal(o[:, :, :i0 + 1], o2[:, :, :i0 + 1])
    assert torch.equal(lse[:, :, :i0 + 1], lse2[:, :, :i0 + 1])
    assert not torch.equal(o[:, :, i0 + 1:], o2[:, :, i0 + 1:])
    # Rows i0+1.. get zero dO: keys past i0 + off are then seen by no row with a gradient.
    do[:, :, i0 + 1:] = 0
    _, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=True, scale=wq.scale)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dk[:, :, i0 + off + 1:]) == 0
    assert torch.count_nonzero(dv[:, :, i0 + off + 1:]) == 0
    assert torch.count_nonzero(dv[:, :, :i0 + off + 1]) > 0


def test_square_call_equals_rectangular_call():
    """attn_fwd_qk with N_q = N_k is attn_fwd: same bits."""
    w = I.custom(1, 2, 384, 128, "bf16", True, seed=12)
    q, k, v = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v"))
    o1, l1 = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
    lib = binding.load()
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    code = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o2.data_ptr(), l2.data_ptr(),
                        1, 2, 384, 128, 1, 1, w.scale,
                        torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert code == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
