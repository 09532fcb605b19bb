"""Failure detection on the GPU without a fault: bounded waits that run out.

A child process sets ATTN_TEST_STALL=1, under which every kernel's TMA producer (the
decode kernel's copying thread) withholds all of its copies: the phases the other roles
wait on never complete, so their waits run out after the pipeline limit
(ATTN_WAIT_LIMIT_CYCLES, read once per process, here 2e5 SM cycles). Each kernel must then
record the site of the first wait that gave up, let the products it issued finish (those
drain waits have their own, fixed bound), release its memory and return. The test checks
that attn_last_kernel_status reports ATTN_ERR_TIMEOUT with a site code of the right
kernel after each call, for the one-CTA-per-item, persistent, CTA-pair, 256-column,
packed-batch and decode kernels, and that the CUDA context is still usable afterwards.

A second check runs the kernels with the limit cut to 64 cycles and nothing withheld. The
waits suspend, and the hardware may hold a suspended wait until its phase completes, so a
call either completes or gives up with its own site code; either way nothing faults or
hangs and the context survives.

Nothing faults, traps or hangs: every wait involved is bounded.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ATTN_ERR_TIMEOUT = 4

CHILD = r"""
import json, sys
import torch
from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

d = int(sys.argv[1])
w = I.custom(1, 2, 768, d, "bf16", True, seed=3)
q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
out = {}
o, lse = binding.attn_fwd(q, k, v, causal=True, scale=w.scale)
out["fwd"] = binding.attn_last_kernel_status()
delta = binding.attn_bwd_preprocess(o, do)
binding.attn_bwd_dkv(q, k, v, lse, delta, do, causal=True, scale=w.scale)
out["dkv"] = binding.attn_last_kernel_status()
binding.attn_bwd_dq(q, k, v, lse, delta, do, causal=True, scale=w.scale)
out["dq"] = binding.attn_last_kernel_status()
qd = I.make_tensor(I.custom(1, 2, 1, d, "bf16", False, seed=4), "q").cuda()
binding.attn_decode(qd, k, v, num_splits=2)
out["decode"] = binding.attn_last_kernel_status()
# a packed batch of two sequences (the PACKED instantiations), host offsets given
cu = torch.tensor([0, 300, 768], dtype=torch.int32)
pq, pk, pv, pdo = (x[0].transpose(0, 1).contiguous() for x in (q, k, v, do))
po, plse = binding.attn_fwd_varlen(pq, pk, pv, cu, cu, 468, 468, causal=True, scale=w.scale)
out["fwd_varlen"] = binding.attn_last_kernel_status()
binding.attn_bwd_varlen(pq, pk, pv, po, plse, pdo, cu, cu, 468, 468, causal=True,
                        scale=w.scale)
out["bwd_varlen"] = binding.attn_last_kernel_status()
torch.cuda.synchronize()
out["after"] = int(torch.arange(10, device="cuda").sum().item())
print(json.dumps(out))
"""

# The site codes of each kernel's waits (kernel * 16 + site, csrc/common.cuh); the dK/dV
# passes of the 256-column backward report the dK/dV kernel's codes.
SITE_RANGE = {"fwd": (0x11, 0x1F), "dq": (0x21, 0x2F), "dkv": (0x31, 0x3F),
              "decode": (0x41, 0x4F), "fwd_varlen": (0x11, 0x1F),
              # the packed backward runs D (no waits), then dK/dV, then dQ: the status
              # word keeps the first wait that ran out, the dK/dV or the dQ kernel's
              "bwd_varlen": (0x21, 0x3F)}


def run_child(d, **env_over):
    env = dict(os.environ, **env_over)
    r = subprocess.run([sys.executable, "-c", CHILD, str(d)], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("d,persistent,pair", [
    (128, "0", "0"), (128, "1", "0"), (128, "1", "1"), (64, "0", "0"), (64, "1", "0"),
    (256, "0", "0"), (256, "1", "0"),
], ids=["d128_one_item", "d128_persistent", "d128_cta_pair", "d64_one_item",
        "d64_persistent", "d256_one_tile", "d256_persistent"])
def test_withheld_copies_make_every_kernel_time_out_and_the_context_survives(
        d, persistent, pair):
    res = run_child(d, ATTN_TEST_STALL="1", ATTN_WAIT_LIMIT_CYCLES="200000",
                    ATTN_FWD_PERSISTENT=persistent, ATTN_BWD_PERSISTENT=persistent,
                    ATTN_FWD_PAIR=pair)
    for name, (lo, hi) in SITE_RANGE.items():
        code, where = res[name]
        assert code == ATTN_ERR_TIMEOUT, (name, code, where)
        assert lo <= where <= hi, (name, hex(where))
    assert res["after"] == 45


@pytest.mark.parametrize("d", [128, 256])
def test_a_tiny_wait_limit_ends_each_call_cleanly(d):
    res = run_child(d, ATTN_WAIT_LIMIT_CYCLES="64")
    for name, (lo, hi) in SITE_RANGE.items():
        code, where = res[name]
        assert code in (0, ATTN_ERR_TIMEOUT), (name, code, where)
        if code == ATTN_ERR_TIMEOUT:
            assert lo <= where <= hi, (name, hex(where))
    assert res["after"] == 45
