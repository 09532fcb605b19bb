"""The seeded input generator: determinism, per-slice regeneration, the spike recipe."""
import math

import torch

from exact_attention_tcgen05_gb300 import inputs as I


def test_slices_regenerate_exactly():
    w = I.custom(2, 3, 40, 16, "bf16", True, 77)
    full = I.make_tensor(w, "q")
    for b in range(2):
        for h in range(3):
            assert torch.equal(full[b, h], I.make_slice(w, b, h, "q"))


def test_tensors_differ_and_are_rounded():
    w = I.custom(1, 2, 64, 32, "fp16", False, 5)
    q, k = I.make_tensor(w, "q"), I.make_tensor(w, "k")
    assert q.dtype == torch.float16 and not torch.equal(q, k)
    assert not torch.equal(q[0, 0], q[0, 1])
    assert abs(q.float().std().item() - 1.0) < 0.1


def test_spike_recipe():
    w = I.BY_NAME["B2_H32_N8192_d64_bf16_full_spiked"]
    pos = I.spike_positions(w)
    assert len(pos) == math.ceil(0.01 * w.N) == len(set(pos.tolist()))
    assert int(pos.min()) >= 3 * w.N // 4 and int(pos.max()) < w.N
    small = I.custom(1, 1, 512, 64, "bf16", False, 1004, qk_gain=4.0, spike=8.0, spike_frac=0.01)
    k = I.make_slice(small, 0, 0, "k").float()
    p = I.spike_positions(small)
    rest = torch.ones(512, dtype=torch.bool)
    rest[p] = False
    assert k[p].mean().item() > 6.0 and abs(k[rest].mean().item()) < 0.5
    assert abs(k[rest].std().item() - 4.0) < 0.3


def test_sampled_slices():
    for w in I.WORKLOADS:
        s = I.sampled_slices(w)
        assert len(s) == min(w.oracle_slices, w.BH) == len(set(s))
        assert s[0] == (0, 0)
        if w.BH > 1:
            assert (w.B - 1, w.H - 1) in s
        assert s == I.sampled_slices(w)
