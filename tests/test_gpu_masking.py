"""Bit-exact masking invariants of the CUDA path (causal mask, ragged tails).

Masked scores must contribute exactly zero, so changing what is masked must leave the
visible results bit-for-bit unchanged.
"""
import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def _run(q, k, v, do, causal, scale):
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("N,d,cut", [(512, 128, 200), (300, 64, 128), (1024, 64, 767)])
def test_future_keys_do_not_leak(N, d, cut):
    """Causal: replacing K, V after position `cut` leaves O, L, dQ of rows <= cut bitwise
    unchanged."""
    w = I.custom(1, 2, N, d, "bf16", True, seed=N + cut)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    base = _run(q, k, v, do, True, w.scale)
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator(device="cpu").manual_seed(99)
    k2[:, :, cut + 1:] = (torch.randn(k2[:, :, cut + 1:].shape, generator=g) * 3).to(k.dtype).cuda()
    v2[:, :, cut + 1:] = (torch.randn(v2[:, :, cut + 1:].shape, generator=g) * 3).to(v.dtype).cuda()
    pert = _run(q, k2, v2, do, True, w.scale)
    for name, a, b in zip(("o", "lse", "dq"), base[:3], pert[:3]):
        assert torch.equal(a[:, :, : cut + 1], b[:, :, : cut + 1]), name


@pytest.mark.parametrize("N,d,j", [(512, 128, 256), (384, 64, 100)])
def test_dkdv_only_from_later_rows(N, d, j):
    """Causal: with dO zero on rows >= j, every key >= j gets dK = dV = 0 exactly
    (its gradient comes from rows i >= key only)."""
    w = I.custom(1, 1, N, d, "fp16", True, seed=3 + j)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    do[:, :, j:] = 0
    _, _, _, dk, dv = _run(q, k, v, do, True, w.scale)
    assert torch.count_nonzero(dk[:, :, j:]) == 0
    assert torch.count_nonzero(dv[:, :, j:]) == 0
    assert torch.count_nonzero(dv[:, :, :j]) > 0


def test_padding_rows_are_not_written():
    """Ragged N: nothing past row N of any slice is touched (outputs live in a larger
    buffer whose tail holds a sentinel)."""
    B, H, N, d = 1, 2, 200, 64
    w = I.custom(B, H, N, d, "bf16", False, seed=8)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    numel = B * H * N * d
    big = torch.full((numel + 4096,), 7.0, dtype=torch.bfloat16, device="cuda")
    o = big[:numel].view(B, H, N, d)
    lse_big = torch.full((B * H * N + 64,), 7.0, dtype=torch.float32, device="cuda")
    lse = lse_big[: B * H * N].view(B, H, N)
    binding.attn_fwd(q, k, v, causal=False, scale=w.scale, o=o, lse=lse)
    torch.cuda.synchronize()
    assert bool((big[numel:] == 7.0).all()) and bool((lse_big[B * H * N:] == 7.0).all())
