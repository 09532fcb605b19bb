"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers such as a plugin inside a host engine that owns all device memory (and hands
out no allocator or workspace), or a serving loop that forbids cudaMalloc after start-up
because it can synchronise the device, cannot provide attn_bwd's workspace. The no-alloc
entry point keeps that scratch (one float32 D value per query row) in a fixed array
inside the library instead. These tests call it through the C ABI and check that it
gives the same bits as attn_bwd, on two calls in a row (the second reuses the array the
first one left behind), and that sizes beyond the array are refused.

This file is collected last on purpose: a failure here leaves every other test run.
"""
import ctypes

import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I



def _noalloc_via_c_abi(w, q, k, v, o, lse, do):
    lib = binding.load()
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    code = lib.attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                dv.data_ptr(), w.B, w.H, w.N, w.d,
                                1 if w.dtype == "bf16" else 0, int(w.causal), w.scale,
                                torch.cuda.current_stream().cuda_stream)
    assert code == binding.ATTN_OK, binding.STATUS_NAMES.get(code, code)
    return dq, dk, dv


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice():
    cases = [I.custom(2, 4, 1000, 128, "bf16", True, seed=41),
             I.custom(1, 3, 515, 64, "fp16", False, seed=42)]
    # two calls in a row, the larger first: the second, smaller one reuses the array the
    # first left behind
    for w in cases:
        q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
        o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
        ref = binding.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
        got = _noalloc_via_c_abi(w, q, k, v, o, lse, do)
        torch.cuda.synchronize()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            # The same kernels on the same D values: the bits must agree exactly, so a
            # wrong array address or D rows left from the larger first call would show.
            assert bool(torch.isfinite(a).all()), name
            assert torch.equal(a, b), (w.name, name)


def test_noalloc_refuses_sizes_beyond_its_array():
    lib = binding.load()
    fake = [0x10000000 + i * (1 << 26) for i in range(9)]
    too_many_rows = binding.NOALLOC_MAX_ROWS + 1  # B * H * N, one row over the limit
    code = lib.attn_bwd_noalloc(*fake, 1, 1, too_many_rows, 64, 1, 0, 0.125, None)
    assert code == 1  # ATTN_ERR_INVALID_ARG, before any CUDA call
    assert lib.attn_bwd_noalloc(*fake, 0, 1, 16, 64, 1, 0, 0.125, None) == 1
