"""The two forward kernels give the same bits.

The library runs the forward either as a persistent kernel (one CTA per SM walking many
(query block, head) items) or as one CTA per item; which one depends on the shape, and
ATTN_FWD_PERSISTENT=0 / 1 forces either. Both compute every tile in the same order with
the same rounding, so O and LSE must agree bit for bit. Each kernel runs in a child process
of its own (the variable is read once per process) on the same seeded inputs.
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
                                 (1, 1, 300, 128, "fp16", False)]:
    w = I.custom(B, H, N, d, dt, causal, seed=N + d)
    q, k, v = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v"))
    o, lse = binding.attn_fwd(q, k, v, causal=causal, scale=w.scale)
    out[w.name] = (o.cpu(), lse.cpu())
wv = I.varlen(2, 128, "bf16", True, seed=3, seqlens_q=(700, 64, 1500, 1))
q, k, v = (I.make_varlen_tensor(wv, t).cuda() for t in ("q", "k", "v"))
cq = torch.tensor(wv.cu_q, dtype=torch.int32, device="cuda")
o, lse = binding.attn_fwd_varlen(q, k, v, cq, cq, wv.max_q, wv.max_k, causal=True)
out["packed"] = (o.cpu(), lse.cpu())
torch.cuda.synchronize()
assert binding.attn_last_kernel_status() == (0, 0)
torch.save(out, sys.argv[2])
"""


def _run(tmp_path, persistent):
    path = str(tmp_path / f"fwd_{persistent}.pt")
    env = dict(os.environ, ATTN_FWD_PERSISTENT=str(persistent))
    subprocess.run([sys.executable, "-c", CHILD, ROOT, path], env=env, check=True,
                   timeout=600)
    return torch.load(path)


def test_persistent_and_one_item_forward_agree_bit_for_bit(tmp_path):
    a = _run(tmp_path, 1)
    b = _run(tmp_path, 0)
    assert a.keys() == b.keys()
    for name in a:
        assert torch.equal(a[name][0], b[name][0]), f"{name}: O differs"
        assert torch.equal(a[name][1], b[name][1]), f"{name}: LSE differs"
