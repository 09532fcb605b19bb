"""Seeded synthetic inputs for the attention workloads.

This module only draws numbers: it holds none of the attention arithmetic, so both
the CUDA path and the fp64 oracle can take their inputs from it without sharing
any computation.

Recipe (one rule for every workload):

* Every (b, h) slice of every tensor (q, k, v, dO) has its own torch CPU generator,
  seeded with ``slice_seed(base_seed, b, h, H, tensor)``. A slice can therefore be
  regenerated alone, which is how the oracle checks sampled heads of the large
  workloads without materialising the others.
* Values are fp32 draws from N(0, 1), multiplied by the workload's ``qk_gain`` for q
  and k, then rounded once to the workload's 16-bit type (round to nearest even,
  torch's cast). The rounded 16-bit values are the inputs of both sides; the oracle
  upcasts them to fp64.
* The softmax-stress workload adds +``spike`` to every feature of a set of
  ceil(``spike_frac`` * N) distinct key positions drawn uniformly from
  [3N/4, N) (one set shared by all heads) before rounding, so that the running
  maximum of late key blocks jumps and the rescale path is exercised.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

_TENSORS = ("q", "k", "v", "do")
_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, 16-bit type, mask and input distribution."""

    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str  # "fp16" | "bf16"
    causal: bool
    seed: int
    qk_gain: float = 1.0
    spike: float = 0.0
    spike_frac: float = 0.0
    oracle_slices: int = 1  # how many (b, h) slices the parity tests check

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def BH(self) -> int:
        return self.B * self.H


# The five workloads, in the order they are quoted.
WORKLOADS = [
    Workload("B1_H1_N256_d128_fp16_full", 1, 1, 256, 128, "fp16", False, 1000, oracle_slices=1),
    Workload("B64_H16_N1024_d64_fp16_causal", 64, 16, 1024, 64, "fp16", True, 1001, oracle_slices=8),
    Workload("B4_H32_N4096_d128_bf16_causal", 4, 32, 4096, 128, "bf16", True, 1002, oracle_slices=4),
    Workload("B1_H16_N16384_d128_bf16_causal", 1, 16, 16384, 128, "bf16", True, 1003, oracle_slices=2),
    Workload("B2_H32_N8192_d64_bf16_full_spiked", 2, 32, 8192, 64, "bf16", False, 1004,
             qk_gain=4.0, spike=8.0, spike_frac=0.01, oracle_slices=2),
]
# Beyond the quoted five: a head dim above 128 (the 256-column kernels), measured beside them.
HEAD_DIM_WORKLOADS = [
    Workload("B4_H16_N4096_d256_bf16_causal", 4, 16, 4096, 256, "bf16", True, 1005,
             oracle_slices=2),
]
BY_NAME = {w.name: w for w in WORKLOADS + HEAD_DIM_WORKLOADS}


def custom(B: int, H: int, N: int, d: int, dtype: str, causal: bool, seed: int,
           qk_gain: float = 1.0, spike: float = 0.0, spike_frac: float = 0.0) -> Workload:
    """A workload outside the quoted five (edge cases: ragged N, tiny N, ...)."""
    name = f"B{B}_H{H}_N{N}_d{d}_{dtype}_{'causal' if causal else 'full'}_s{seed}"
    return Workload(name, B, H, N, d, dtype, causal, seed, qk_gain, spike, spike_frac)


def slice_seed(base_seed: int, b: int, h: int, H: int, tensor: str) -> int:
    """Generator seed of one (b, h) slice of one tensor."""
    return (base_seed * 1_000_003 + (b * H + h)) * 8 + _TENSORS.index(tensor)


def spike_positions(w: Workload) -> torch.Tensor:
    """Key positions that receive the spike (empty when the workload has none)."""
    if w.spike == 0.0 or w.spike_frac == 0.0:
        return torch.empty(0, dtype=torch.long)
    lo = (3 * w.N) // 4
    count = min(w.N - lo, math.ceil(w.spike_frac * w.N))
    g = torch.Generator().manual_seed(w.seed * 7919 + 17)
    return torch.randperm(w.N - lo, generator=g)[:count] + lo


def make_slice(w: Workload, b: int, h: int, tensor: str,
               spikes: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One [N, d] slice, rounded to the workload's 16-bit type, on the CPU."""
    g = torch.Generator().manual_seed(slice_seed(w.seed, b, h, w.H, tensor))
    x = torch.randn(w.N, w.d, generator=g, dtype=torch.float32)
    if tensor in ("q", "k") and w.qk_gain != 1.0:
        x = x * w.qk_gain
    if tensor == "k" and w.spike != 0.0:
        pos = spike_positions(w) if spikes is None else spikes
        x[pos] += w.spike
    return x.to(w.torch_dtype)


def make_tensor(w: Workload, tensor: str) -> torch.Tensor:
    """The full [B, H, N, d] tensor on the CPU (contiguous)."""
    spikes = spike_positions(w) if tensor == "k" else None
    out = torch.empty(w.B, w.H, w.N, w.d, dtype=w.torch_dtype)
    for b in range(w.B):
        for h in range(w.H):
            out[b, h] = make_slice(w, b, h, tensor, spikes)
    return out


def make_tensor_cuda(w: Workload, tensor: str) -> torch.Tensor:
    """The full [B, H, N, d] tensor drawn directly on the current CUDA device, for
    workloads too large to draw on the host (gigabytes of K/V): one CUDA generator per
    tensor, seeded from the workload seed and the tensor name, fp32 N(0, 1) values times
    qk_gain for q and k, then one rounding to the 16-bit type. Spikes are not applied.
    The oracle reads the same rounded values back with to_f64."""
    g = torch.Generator(device="cuda").manual_seed(slice_seed(w.seed, 0, 0, 1, tensor))
    x = torch.randn(w.B, w.H, w.N, w.d, generator=g, device="cuda", dtype=torch.float32)
    if tensor in ("q", "k") and w.qk_gain != 1.0:
        x.mul_(w.qk_gain)
    return x.to(w.torch_dtype)


def sampled_slices(w: Workload, count: Optional[int] = None) -> list[tuple[int, int]]:
    """Seeded choice of (b, h) slices without replacement; always holds the first and
    the last slice."""
    count = w.oracle_slices if count is None else count
    count = min(count, w.BH)
    first, last = 0, w.BH - 1
    chosen = [first] if count >= 1 else []
    if count >= 2 and last != first:
        chosen.append(last)
    rest = [i for i in range(w.BH) if i not in chosen]
    g = torch.Generator().manual_seed(w.seed * 104729 + 3)
    perm = torch.randperm(len(rest), generator=g).tolist()
    chosen += [rest[i] for i in perm[: max(0, count - len(chosen))]]
    return [(i // w.H, i % w.H) for i in chosen]


def to_f64(x: torch.Tensor):
    """Exact upcast of rounded 16-bit values to a float64 numpy array."""
    return x.detach().to("cpu").to(torch.float64).numpy()


# ------------------------------------------------------------------------------------
# Packed variable-length batches: sequences one after another along the token axis,
# q, k, v, dO as [total, H, d], boundaries as cu_seqlens (B + 1 cumulative lengths).
# ------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of sequences of different lengths (query and key lengths per
    sequence), 16-bit type, mask and seed."""

    name: str
    H: int
    d: int
    dtype: str
    causal: bool
    seed: int
    seqlens_q: tuple
    seqlens_k: tuple

    @property
    def torch_dtype(self) -> torch.dtype:
        return _DTYPES[self.dtype]

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def B(self) -> int:
        return len(self.seqlens_q)

    @staticmethod
    def _cu(lengths) -> list[int]:
        out = [0]
        for n in lengths:
            out.append(out[-1] + int(n))
        return out

    @property
    def cu_q(self) -> list[int]:
        return self._cu(self.seqlens_q)

    @property
    def cu_k(self) -> list[int]:
        return self._cu(self.seqlens_k)

    @property
    def total_q(self) -> int:
        return sum(self.seqlens_q)

    @property
    def total_k(self) -> int:
        return sum(self.seqlens_k)

    @property
    def max_q(self) -> int:
        return max(self.seqlens_q)

    @property
    def max_k(self) -> int:
        return max(self.seqlens_k)


def length_mix(total: int, lo: int, hi: int, seed: int) -> tuple:
    """Seeded sequence lengths drawn uniformly from [lo, hi] until they add up to
    `total` (the last one is cut to fit; a cut below 1 is dropped)."""
    g = torch.Generator().manual_seed(seed * 7 + 5)
    out = []
    left = total
    while left > 0:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        out.append(min(n, left))
        left -= out[-1]
    return tuple(out)


def varlen(H: int, d: int, dtype: str, causal: bool, seed: int, seqlens_q, seqlens_k=None,
           name: Optional[str] = None) -> VarlenWorkload:
    """A packed workload with the given per-sequence lengths (keys = queries if absent)."""
    seqlens_q = tuple(int(n) for n in seqlens_q)
    seqlens_k = seqlens_q if seqlens_k is None else tuple(int(n) for n in seqlens_k)
    if len(seqlens_k) != len(seqlens_q):
        raise ValueError("one key length per sequence")
    if name is None:
        name = (f"varlen_B{len(seqlens_q)}_H{H}_T{sum(seqlens_q)}_d{d}_{dtype}_"
                f"{'causal' if causal else 'full'}_s{seed}")
    return VarlenWorkload(name, H, d, dtype, causal, seed, seqlens_q, seqlens_k)


# The packed benchmark batch: 16384 tokens (the token count of B4 x N4096) in sequences
# of 512 .. 4096 tokens, 32 heads, d = 128, bf16, causal.
VARLEN_BENCH = varlen(32, 128, "bf16", True, 1010, length_mix(16384, 512, 4096, 1010),
                      name="varlen_H32_T16384_len512-4096_d128_bf16_causal")


def make_varlen_tensor(w: VarlenWorkload, tensor: str) -> torch.Tensor:
    """The packed [total, H, d] tensor on the CPU: rows cu[b] .. cu[b+1] of head h come
    from the generator of slice (b, h) of `tensor` (as for the dense workloads: fp32
    N(0, 1), one rounding to the 16-bit type)."""
    lengths = w.seqlens_q if tensor in ("q", "do") else w.seqlens_k
    cu = VarlenWorkload._cu(lengths)
    out = torch.empty(cu[-1], w.H, w.d, dtype=w.torch_dtype)
    for b, n in enumerate(lengths):
        for h in range(w.H):
            g = torch.Generator().manual_seed(slice_seed(w.seed, b, h, w.H, tensor))
            out[cu[b]:cu[b + 1], h] = torch.randn(n, w.d, generator=g,
                                                  dtype=torch.float32).to(w.torch_dtype)
    return out
