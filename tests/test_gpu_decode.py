"""GPU parity of split-KV decoding (attn_decode_partial / attn_decode_merge / attn_decode)
against the fp64 decode oracle (oracle/decode.py), on the same seeded inputs.

Tolerances: O max-abs 1e-2 plus half an ulp of the output dtype at |O| (as for the
forward), L 1e-3. The per-split records are compared too: m 1e-3, l and O~ to 1e-3 of
their scale (the kernel keeps them in fp32 with exp2.approx weights, and never rounds
the weights to 16 bits).
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I
import oracle.decode as OD

from parity import o_error

pytestmark = pytest.mark.gpu

L_TOL = 1e-3
REC_TOL = 1e-3


def _tensors(B, H, Nk, d, dtype, seed, qk_gain=1.0, on_device=False):
    """q [B, H, 1, d] and k, v [B, H, Nk, d] from the seeded input generators (drawn on
    the device for the large workload)."""
    wq = I.custom(B, H, 1, d, dtype, False, seed=seed, qk_gain=qk_gain)
    wk = I.custom(B, H, Nk, d, dtype, False, seed=seed + 1, qk_gain=qk_gain)
    make = I.make_tensor_cuda if on_device else (lambda w, t: I.make_tensor(w, t).cuda())
    return make(wq, "q"), make(wk, "k"), make(wk, "v")


def _half_ulp(x, dtype):
    mant = 7 if dtype == torch.bfloat16 else 10
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return 0.5 * np.exp2(e - mant)


def _check_slice(q, k, v, o, lse, parts, b, h, scale, splits):
    qd, kd, vd = (I.to_f64(x[b, h].cpu()) for x in (q, k, v))
    ref_o, ref_l, ref_parts = OD.decode(qd[0], kd, vd, scale, splits)
    got_o = o[b, h, 0].float().cpu().double().numpy()
    r = o_error(got_o, ref_o, o.dtype)
    assert r["o_excess"] <= 0, f"O error {r['o_max']:.3e}"
    assert abs(float(lse[b, h]) - ref_l) <= L_TOL, f"L {float(lse[b, h])} vs {ref_l}"
    if parts is None:
        return
    d = kd.shape[1]
    rec = parts[b, h].cpu().double().numpy()
    for s, (m_r, l_r, u_r) in enumerate(ref_parts):
        if m_r == -math.inf:
            assert rec[s, d] == -math.inf and rec[s, d + 1] == 0.0
            assert np.all(rec[s, :d] == 0.0)
            continue
        assert abs(rec[s, d] - m_r) <= REC_TOL, (s, rec[s, d], m_r)
        assert abs(rec[s, d + 1] / l_r - 1.0) <= REC_TOL
        scale_u = max(1e-6, np.abs(u_r).max())
        assert np.abs(rec[s, :d] - u_r).max() <= REC_TOL * scale_u


CASES = [
    # B, H, Nk, d, dtype, splits
    (1, 2, 1, 128, "bf16", 1),
    (1, 2, 63, 64, "fp16", 1),
    (2, 1, 64, 128, "bf16", 3),     # more splits than sub-blocks: empty splits
    (1, 3, 65, 128, "fp16", 2),
    (2, 2, 1000, 64, "bf16", 7),
    (1, 2, 4113, 128, "bf16", 16),  # ragged last sub-block, several sub-blocks per split
    (1, 1, 3000, 128, "fp16", 1),   # one split over many sub-blocks (ring reuse)
    (1, 2, 1, 256, "bf16", 1),      # d = 256: one stage of one sub-block
    (2, 1, 64, 256, "fp16", 3),
    (1, 2, 4113, 256, "bf16", 16),
    (1, 1, 3000, 256, "fp16", 1),
]


@pytest.mark.parametrize("B,H,Nk,d,dtype,splits", CASES)
def test_decode_matches_oracle(B, H, Nk, d, dtype, splits):
    q, k, v = _tensors(B, H, Nk, d, dtype, seed=100 + Nk + splits)
    scale = 1.0 / math.sqrt(d)
    parts = binding.attn_decode_partial(q, k, v, scale=scale, num_splits=splits)
    o, lse = binding.attn_decode_merge(parts, q.dtype)
    o2, lse2 = binding.attn_decode(q, k, v, scale=scale, num_splits=splits)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
    for b in range(B):
        for h in range(H):
            _check_slice(q, k, v, o, lse, parts, b, h, scale, splits)


def test_decode_spiky_scores():
    """Scores spread over a wide range (q, k x4; one key +8): the running max moves."""
    B, H, Nk, d = 1, 2, 2048, 128
    q, k, v = _tensors(B, H, Nk, d, "bf16", seed=7, qk_gain=4.0)
    k[:, :, 1500] += 8
    scale = 1.0 / math.sqrt(d)
    o, lse = binding.attn_decode(q, k, v, scale=scale, num_splits=5)
    parts = binding.attn_decode_partial(q, k, v, scale=scale, num_splits=5)
    torch.cuda.synchronize()
    for h in range(H):
        _check_slice(q, k, v, o, lse, parts, 0, h, scale, 5)


def test_merge_kernel_against_oracle_merge():
    """The merge kernel applied to the GPU's records equals the oracle's merge of the
    same records (pins the merge alone, independent of the partial kernel's error)."""
    B, H, Nk, d, splits = 2, 2, 5000, 64, 9
    q, k, v = _tensors(B, H, Nk, d, "fp16", seed=31)
    parts = binding.attn_decode_partial(q, k, v, scale=0.125, num_splits=splits)
    o, lse = binding.attn_decode_merge(parts, q.dtype)
    torch.cuda.synchronize()
    rec = parts.cpu().double().numpy()
    for b in range(B):
        for h in range(H):
            states = [(rec[b, h, s, d], rec[b, h, s, d + 1], rec[b, h, s, :d])
                      for s in range(splits)]
            ref_o, ref_l = OD.finish(*OD.merge_states(states))
            got = o[b, h, 0].float().cpu().double().numpy()
            assert np.all(np.abs(got - ref_o) <= 1e-5 + _half_ulp(ref_o, o.dtype))
            assert abs(float(lse[b, h]) - ref_l) <= 1e-5


def test_split_record_depends_only_on_its_keys():
    """Changing keys outside split s leaves split s's record bit-for-bit unchanged."""
    B, H, Nk, d, splits = 1, 2, 1024, 128, 4  # splits of 256 keys
    q, k, v = _tensors(B, H, Nk, d, "bf16", seed=5)
    base = binding.attn_decode_partial(q, k, v, scale=0.09, num_splits=splits).clone()
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 512:] = -k2[:, :, 512:] * 3
    v2[:, :, 512:] = v2[:, :, 512:] + 1
    pert = binding.attn_decode_partial(q, k2, v2, scale=0.09, num_splits=splits)
    torch.cuda.synchronize()
    assert torch.equal(base[:, :, :2], pert[:, :, :2])
    assert not torch.equal(base[:, :, 2:], pert[:, :, 2:])


def test_decode_split_count_does_not_change_the_answer():
    B, H, Nk, d = 2, 2, 3000, 128
    q, k, v = _tensors(B, H, Nk, d, "bf16", seed=17)
    outs = [binding.attn_decode(q, k, v, num_splits=s) for s in (1, 2, 5, 47)]
    torch.cuda.synchronize()
    for o, lse in outs[1:]:
        assert (o.float() - outs[0][0].float()).abs().max().item() <= 1e-2
        assert (lse - outs[0][1]).abs().max().item() <= 1e-4


def test_decode_bench_workload_sampled():
    """The decode bench workload (B8 H32 Nk32768 d128 bf16, default splits) on sampled
    slices, in the launch configuration bench.py times."""
    B, H, Nk, d = 8, 32, 32768, 128
    q, k, v = _tensors(B, H, Nk, d, "bf16", seed=2024, on_device=True)
    splits = binding.attn_decode_splits(B, H, Nk)
    o, lse = binding.attn_decode(q, k, v, num_splits=splits)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (3, 17), (7, 31)]:
        _check_slice(q, k, v, o, lse, None, b, h, 1.0 / math.sqrt(d), splits)
