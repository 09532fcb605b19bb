"""attn_step_host (host buffers in and out, copies overlapped with the kernels) gives the
same bits as attn_fwd + attn_bwd on device tensors: every (b, h) slice is computed by the
same kernels, whatever chunk it falls in."""
import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,H,N,d,dtype,causal,chunks", [
    (2, 3, 300, 128, "bf16", True, 4),
    (1, 2, 256, 64, "fp16", False, 1),
    (2, 2, 513, 128, "bf16", False, 3),
    (1, 3, 128, 64, "bf16", True, 9),   # more chunks than slices (clamped)
    (1, 3, 300, 256, "bf16", True, 2),  # the 256-column kernels
    (2, 3, 203, 128, "fp16", False, 5),  # N % 4 = 3: rows of L not 16-byte multiples
])
def test_step_host_matches_device_path(B, H, N, d, dtype, causal, chunks):
    w = I.custom(B, H, N, d, dtype, causal, seed=N + chunks)
    host = {t: I.make_tensor(w, t).pin_memory() for t in ("q", "k", "v", "do")}
    out = {n: torch.empty(host["q"].shape, dtype=host["q"].dtype).pin_memory()
           for n in ("o", "dq", "dk", "dv")}
    lse_h = torch.empty(B, H, N, dtype=torch.float32).pin_memory()
    scratch = torch.empty(binding.attn_step_host_scratch_bytes(B, H, N, d, chunks),
                          dtype=torch.uint8, device="cuda")
    binding.attn_step_host(host["q"], host["k"], host["v"], host["do"], out["o"], lse_h,
                           out["dq"], out["dk"], out["dv"], scratch, causal=causal,
                           scale=w.scale, chunks=chunks)
    torch.cuda.synchronize()
    dev = {t: x.cuda() for t, x in host.items()}
    o, lse = binding.attn_fwd(dev["q"], dev["k"], dev["v"], causal=causal, scale=w.scale)
    dq, dk, dv = binding.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                                  causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert torch.equal(out[name], ref.cpu()), name
    assert torch.equal(lse_h, lse.cpu())


def test_step_host_back_to_back_calls():
    """Two calls queued on one stream with no synchronisation between them, on different
    inputs and with different chunk counts, reuse the side streams and events: each gives
    the bits of the device path for its own inputs."""
    B, H, N, d = 2, 4, 384, 128
    runs = []
    for seed, chunks in ((5, 6), (6, 3)):
        w = I.custom(B, H, N, d, "bf16", True, seed=seed)
        host = {t: I.make_tensor(w, t).pin_memory() for t in ("q", "k", "v", "do")}
        out = {n: torch.empty(host["q"].shape, dtype=host["q"].dtype).pin_memory()
               for n in ("o", "dq", "dk", "dv")}
        lse_h = torch.empty(B, H, N, dtype=torch.float32).pin_memory()
        scratch = torch.empty(binding.attn_step_host_scratch_bytes(B, H, N, d, chunks),
                              dtype=torch.uint8, device="cuda")
        binding.attn_step_host(host["q"], host["k"], host["v"], host["do"], out["o"], lse_h,
                               out["dq"], out["dk"], out["dv"], scratch, causal=True,
                               scale=w.scale, chunks=chunks)
        runs.append((w, host, out, lse_h, scratch))
    torch.cuda.synchronize()
    for w, host, out, lse_h, _ in runs:
        dev = {t: x.cuda() for t, x in host.items()}
        o, lse = binding.attn_fwd(dev["q"], dev["k"], dev["v"], causal=True, scale=w.scale)
        dq, dk, dv = binding.attn_bwd(dev["q"], dev["k"], dev["v"], o, lse, dev["do"],
                                      causal=True, scale=w.scale)
        torch.cuda.synchronize()
        for name, ref in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            assert torch.equal(out[name], ref.cpu()), name
        assert torch.equal(lse_h, lse.cpu())
