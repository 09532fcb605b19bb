"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI on seeded
inputs, run the fp64 oracle on the same rounded inputs, and compare.

Tolerances (the bar the CUDA path must meet against the oracle):
  O    |O_gpu - O_ref| <= 1e-2 wherever |O_ref| < 2. Where |O_ref| >= 2 the output
       type's own storage rounding comes on top: 1e-2 + half an ulp of the output type
       at |O_ref| (bf16: 0.0078 for |O| in [2, 4), 0.0156 in [4, 8)). Below 2 half an
       ulp is at most 0.0039 and the flat 1e-2 holds on its own. The CPU emulation in
       test_rounding_emulation.py shows why the allowance exists: a kernel that rounds
       P to the input type before P V, as "Triton 05: Flash Attention" prescribes
       (section 코드 라인별 설명 (Forward), step 5, p.to(v.dtype)), stays within 1e-2
       before storage but exceeds it at |O| >= 2 once O is stored in bf16.
  LSE  max-abs <= 1e-3;
  dQ, dK, dV  relative Frobenius error <= 3e-2 per (b, h) slice, with an absolute
       floor of 1e-5 RMS for gradients that vanish exactly (e.g. N = 1 causal, where
       dS = P (dP - D) = 0, so dQ = dK = 0 and only fp32 rounding is left).

Every comparison is also recorded (see RECORD) so that the test session can print the
raw errors per workload at its end.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle.attention as OA
from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

O_TOL = 1e-2
O_STORAGE_FROM = 2.0  # |O_ref| from which half an output ulp is allowed on top of O_TOL
LSE_TOL = 1e-3
GRAD_TOL = 3e-2
GRAD_RMS_FLOOR = 1e-5


@dataclasses.dataclass
class GpuRun:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor
    o: torch.Tensor
    lse: torch.Tensor
    dq: torch.Tensor
    dk: torch.Tensor
    dv: torch.Tensor


def make_inputs(w: I.Workload, device="cuda"):
    return tuple(I.make_tensor(w, t).to(device) for t in ("q", "k", "v", "do"))


def run_gpu(w: I.Workload, tensors=None, backward=True) -> GpuRun:
    q, k, v, do = make_inputs(w) if tensors is None else tensors
    o, lse = binding.attn_fwd(q, k, v, causal=w.causal, scale=w.scale)
    if backward:
        dq, dk, dv = binding.attn_bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
    else:
        dq = dk = dv = None
    torch.cuda.synchronize()
    return GpuRun(q, k, v, do, o, lse, dq, dk, dv)


def ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    mant = 7 if dtype == torch.bfloat16 else 10
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    return np.exp2(e - mant)


def o_error(o_gpu: np.ndarray, o_ref: np.ndarray, dtype) -> dict:
    """Raw max error, max excess over the bound (pass iff <= 0), and how many elements
    needed the storage allowance (error above O_TOL, possible only at |O_ref| >= 2)."""
    err = np.abs(o_gpu - o_ref)
    big = np.abs(o_ref) >= O_STORAGE_FROM
    allowed = np.where(big, O_TOL + 0.5 * ulp(o_ref, dtype), O_TOL)
    small_err = err[~big]
    return {"o_max": float(err.max()),
            "o_max_below2": float(small_err.max()) if small_err.size else 0.0,
            "o_excess": float((err - allowed).max()),
            "o_allowance_used": int((err > O_TOL).sum())}


def rel_fro(a: np.ndarray, b: np.ndarray) -> float:
    """||a - b||_F / max(||b||_F, floor * sqrt(numel))."""
    floor = GRAD_RMS_FLOOR * np.sqrt(b.size)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), floor))


def compare_slice(w: I.Workload, run: GpuRun, b: int, h: int, backward=True) -> dict:
    """Oracle on slice (b, h) from the same rounded inputs; returns the errors."""
    q, k, v, do = (I.to_f64(x[b, h]) for x in (run.q, run.k, run.v, run.do))
    if backward:
        ref = OA.attention_backward(q, k, v, do, w.causal, w.scale)
    else:
        o_ref, lse_ref = OA.attention_forward(q, k, v, w.causal, w.scale)
        ref = dict(o=o_ref, lse=lse_ref)
    res = o_error(I.to_f64(run.o[b, h]), ref["o"], w.torch_dtype)
    res["lse_max"] = float(np.abs(run.lse[b, h].double().cpu().numpy() - ref["lse"]).max())
    if backward:
        for name in ("dq", "dk", "dv"):
            res[name] = rel_fro(I.to_f64(getattr(run, name)[b, h]), ref[name])
    return res


# Comparisons made in this session: {label: {"slices": n, "o_max": ..., ...}} (worst
# values over the slices), printed by the terminal-summary hook in conftest.py.
RECORD: dict = {}


def record(label: str, res: dict) -> None:
    r = RECORD.setdefault(label, {"slices": 0})
    r["slices"] += 1
    for key, val in res.items():
        if key == "o_allowance_used":
            r[key] = r.get(key, 0) + val
        else:
            r[key] = max(r.get(key, val), val)


def assert_within(res: dict, where: str) -> None:
    assert res["o_excess"] <= 0.0, f"{where}: O error {res['o_max']:.3e} above bound"
    assert res["lse_max"] <= LSE_TOL, f"{where}: LSE error {res['lse_max']:.3e}"
    for name in ("dq", "dk", "dv"):
        if name in res:
            assert res[name] <= GRAD_TOL, f"{where}: {name} rel. Frobenius {res[name]:.3e}"


def all_finite(run: GpuRun) -> bool:
    ts = [run.o, run.lse] + ([run.dq, run.dk, run.dv] if run.dq is not None else [])
    return all(bool(torch.isfinite(t).all()) for t in ts)
