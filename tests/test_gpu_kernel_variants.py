"""The persistent and the one-item kernels give the same bits.

The forward (at every head dim), dK/dV and dQ kernels each exist as a persistent kernel (one
CTA per SM walking many work items) and as one CTA per item; which one runs depends on the shape, and
ATTN_FWD_PERSISTENT / ATTN_BWD_PERSISTENT = 0 / 1 force either. The 128-column forward also
exists on CTA pairs (ATTN_FWD_PAIR = 1). Both compute every tile in
the same order with the same rounding, so O, LSE, dQ, dK and dV must agree bit for bit.
Each setting runs in a child process of its own (the variables are read once per process)
on the same seeded inputs.
"""
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I
out = {}
for (B, H, N, d, dt, causal) in [(2, 3, 1000, 128, "bf16", True), (1, 4, 777, 64, "fp16", False),
                                 (3, 2, 2100, 64, "bf16", True), (1, 2, 4096, 64, "bf16", False),
                                 (1, 1, 300, 128, "fp16", False),
                                 # more causal items than SMs: the forward's scheduled order
                                 (4, 16, 1280, 128, "bf16", True), (8, 8, 1024, 64, "fp16", True),
                                 # head dims above 128: the 256-column forward
                                 (2, 3, 1000, 256, "bf16", True), (1, 2, 777, 192, "fp16", False),
                                 (4, 8, 1280, 256, "bf16", True)]:
    w = I.custom(B, H, N, d, dt, causal, seed=N + d)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=w.scale)
    dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=causal, scale=w.scale)
    out[w.name] = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
wv = I.varlen(2, 128, "bf16", True, seed=3, seqlens_q=(700, 64, 1500, 1))
q, k, v, do = (I.make_varlen_tensor(wv, t).cuda() for t in ("q", "k", "v", "do"))
cq = torch.tensor(wv.cu_q, dtype=torch.int32, device="cuda")
o, lse = binding.attn_fwd_varlen(q, k, v, cq, cq, wv.max_q, wv.max_k, causal=True)
dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, cq, cq, wv.max_q, wv.max_k,
                                     causal=True)
out["packed"] = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
wv = I.varlen(3, 64, "fp16", True, seed=4, seqlens_q=(300, 1, 900, 129, 40))
q, k, v, do = (I.make_varlen_tensor(wv, t).cuda() for t in ("q", "k", "v", "do"))
cq = torch.tensor(wv.cu_q, dtype=torch.int32, device="cuda")
o, lse = binding.attn_fwd_varlen(q, k, v, cq, cq, wv.max_q, wv.max_k, causal=True)
dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, cq, cq, wv.max_q, wv.max_k,
                                     causal=True)
out["packed_d64"] = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
wv = I.varlen(2, 256, "bf16", True, seed=6, seqlens_q=(500, 1, 900, 129))
q, k, v, do = (I.make_varlen_tensor(wv, t).cuda() for t in ("q", "k", "v", "do"))
cq = torch.tensor(wv.cu_q, dtype=torch.int32, device="cuda")
o, lse = binding.attn_fwd_varlen(q, k, v, cq, cq, wv.max_q, wv.max_k, causal=True)
dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, cq, cq, wv.max_q, wv.max_k,
                                     causal=True)
out["packed_d256"] = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
# N_q = 640 against N_k = 1000 (bottom-right causal), more items than SMs in every kernel:
# the scheduled orders with an offset
wq = I.custom(4, 40, 640, 64, "bf16", True, seed=21)
wk = I.custom(4, 40, 1000, 64, "bf16", True, seed=22)
q, do = (I.make_tensor(wq, t).cuda() for t in ("q", "do"))
k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
o, lse = binding.attn_fwd(q, k, v, causal=True, scale=wq.scale)
dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=True, scale=wq.scale)
out["rect"] = tuple(x.cpu() for x in (o, lse, dq, dk, dv))
torch.cuda.synchronize()
assert binding.attn_last_kernel_status() == (0, 0)
torch.save(out, sys.argv[2])
"""


def _run(tmp_path, persistent, pair=0):
    path = str(tmp_path / f"run_{persistent}_{pair}.pt")
    env = dict(os.environ, ATTN_FWD_PERSISTENT=str(persistent),
               ATTN_BWD_PERSISTENT=str(persistent), ATTN_FWD_PAIR=str(pair))
    subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, check=True,
                   timeout=600)
    return torch.load(path)


def test_persistent_and_one_item_kernels_agree_bit_for_bit(tmp_path):
    a = _run(tmp_path, 1)
    b = _run(tmp_path, 0)
    assert a.keys() == b.keys()
    for name in a:
        for what, x, y in zip(("O", "LSE", "dQ", "dK", "dV"), a[name], b[name]):
            assert torch.equal(x, y), f"{name}: {what} differs"


def test_cta_pair_forward_agrees_bit_for_bit(tmp_path):
    """ATTN_FWD_PAIR = 1: the 128-column forward runs on CTA pairs (csrc/fwd_pair.cuh),
    tcgen05 MMAs with .cta_group::2 over two SMs. Each S and P V element is computed from
    the same operands in the same order as in the one-CTA kernel, so every output of the
    cases above (dense d = 128 causal and full, ragged, more items than clusters, a packed
    batch) must be the same bits; the d = 64 cases run the same kernels in both."""
    a = _run(tmp_path, 1, pair=1)
    b = _run(tmp_path, 1, pair=0)
    assert a.keys() == b.keys()
    for name in a:
        for what, x, y in zip(("O", "LSE", "dQ", "dK", "dV"), a[name], b[name]):
            assert torch.equal(x, y), f"{name}: {what} differs"
