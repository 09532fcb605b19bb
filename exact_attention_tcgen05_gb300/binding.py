"""ctypes binding of libattn.so: argument marshalling only.

Every function here checks that the tensors are what the C ABI expects (CUDA,
contiguous, [B, H, N, d], one 16-bit dtype), allocates outputs with torch when the
caller passes none, and calls the library on `stream` (default: torch's current
stream). With a stream given, everything the function allocates or copies (outputs,
workspaces, cu_seqlens uploaded from the CPU) is made on that stream, so the caching
allocator cannot hand that memory to other work while the kernels still use it. All arithmetic
runs in the library's kernels; there is no fallback of any kind: if the library is
missing or fails, these functions raise.
"""
from __future__ import annotations

import ctypes
import functools
import inspect
import math
import os
from typing import Optional

import torch

from .build import LIB_PATH

ATTN_OK = 0
STATUS_NAMES = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
                3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_TIMEOUT"}
_DTYPE_CODES = {torch.float16: 0, torch.bfloat16: 1}

# Public entry points declared in include/attn.h and their ctypes signatures.
_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_fwd_qk": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_qk": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                         _P]),
    "attn_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "attn_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                             _I, _F, _P]),
    "attn_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I,
                             _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_varlen_workspace_bytes": (ctypes.c_size_t, [_I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_preprocess": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_bwd_dkv": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_dq": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "attn_bwd_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                              _P]),
    "attn_step_host_scratch_bytes": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "attn_step_host": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _I, _I, _I,
                            _I, _I, _I, _F, _I, _P]),
    "attn_decode_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "attn_decode_splits": (_I, [_I, _I, _I]),
    "attn_decode_partial": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_decode_merge": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "attn_status_str": (ctypes.c_char_p, [_I]),
    "attn_last_kernel_status": (_I, [_P, ctypes.POINTER(_I)]),
}

_lib: Optional[ctypes.CDLL] = None


class AttnError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(code, code)}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libattn.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                f"g.build()\"` (nvcc, sm_103a). There is no fallback implementation.")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _on_launch_stream(fn):
    """Runs fn with its `stream` argument (if given) as torch's current stream, so that
    the tensors fn allocates and the copies it makes are ordered with its launches."""
    sig = inspect.signature(fn)

    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        stream = sig.bind_partial(*args, **kwargs).arguments.get("stream")
        if stream is None:
            return fn(*args, **kwargs)
        with torch.cuda.stream(stream):
            return fn(*args, **kwargs)
    return wrapper


def _stream_handle(stream: Optional[torch.cuda.Stream]) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn: str, code: int) -> None:
    if code != ATTN_OK:
        raise AttnError(fn, code)


def _shape_of(x: torch.Tensor, name: str) -> tuple[int, int, int, int]:
    if not isinstance(x, torch.Tensor) or x.dim() != 4:
        raise ValueError(f"{name} must be a [B, H, N, d] tensor")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if x.dtype not in _DTYPE_CODES:
        raise ValueError(f"{name} must be float16 or bfloat16")
    return tuple(x.shape)  # type: ignore[return-value]


def _same(ref: torch.Tensor, x: torch.Tensor, name: str) -> None:
    _shape_of(x, name)
    if x.shape != ref.shape or x.dtype != ref.dtype or x.device != ref.device:
        raise ValueError(f"{name} must match q in shape, dtype and device")


def _keys_like(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> int:
    """N_k of k and v, which match q in B, H, d, dtype and device and each other."""
    B, H, _, d = q.shape
    Bk, Hk, Nk, dk = _shape_of(k, "k")
    if (Bk, Hk, dk) != (B, H, d) or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k must be [B, H, N_k, d] with q's dtype and device")
    _same(k, v, "v")
    return Nk


def _lse_like(q: torch.Tensor, x: Optional[torch.Tensor], name: str) -> torch.Tensor:
    B, H, N, _ = q.shape
    if x is None:
        return torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if x.shape != (B, H, N) or x.dtype != torch.float32 or not x.is_contiguous() \
            or x.device != q.device:
        raise ValueError(f"{name} must be a contiguous float32 [B, H, N] tensor on q's device")
    return x


@_on_launch_stream
def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> tuple[torch.Tensor, torch.Tensor]:
    """O = softmax(scale q k^T [causal]) v and the natural-log LSE, via libattn.so.
    k and v may hold more rows than q (N_k >= N_q when causal; bottom-right aligned)."""
    B, H, N, d = _shape_of(q, "q")
    Nk = _keys_like(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    if o is None:
        o = torch.empty_like(q)
    else:
        _same(q, o, "o")
    lse = _lse_like(q, lse, "lse")
    with torch.cuda.device(q.device):
        code = load().attn_fwd_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), B, H, N, Nk, d, _DTYPE_CODES[q.dtype],
                                  int(causal), scale, _stream_handle(stream))
    _check("attn_fwd_qk", code)
    return o, lse


def attn_bwd_workspace_bytes(B: int, H: int, N: int) -> int:
    return int(load().attn_bwd_workspace_bytes(B, H, N))


@_on_launch_stream
def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
             lse: torch.Tensor, do: torch.Tensor, causal: bool = False,
             scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None
             ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dq, dk, dv of sum(do * o), recomputing P from lse, via libattn.so. k and v may
    hold more rows than q (as in attn_fwd)."""
    B, H, N, d = _shape_of(q, "q")
    Nk = _keys_like(q, k, v)
    for name, x in (("o", o), ("do", do)):
        _same(q, x, name)
    lse = _lse_like(q, lse, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _same(q, dq, "dq")
    _same(k, dk, "dk")
    _same(k, dv, "dv")
    workspace = _lse_like(q, workspace, "workspace")
    with torch.cuda.device(q.device):
        code = load().attn_bwd_qk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), workspace.data_ptr(), B, H, N, Nk, d,
                                  _DTYPE_CODES[q.dtype], int(causal), scale,
                                  _stream_handle(stream))
    _check("attn_bwd_qk", code)
    return dq, dk, dv


NOALLOC_MAX_ROWS = 4194304  # ATTN_NOALLOC_MAX_ROWS in include/attn.h


@_on_launch_stream
def attn_bwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                     lse: torch.Tensor, do: torch.Tensor, causal: bool = False,
                     scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
                     dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None
                     ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """attn_bwd for callers that cannot allocate a workspace: the library's own
    fixed-size scratch array holds the per-row D values (B*H*N <= NOALLOC_MAX_ROWS).
    Calls that overlap on the GPU share that array and race; serialise them. This
    wrapper still lets torch allocate dq, dk, dv when they are not passed in."""
    B, H, N, d = _shape_of(q, "q")
    for name, x in (("k", k), ("v", v), ("o", o), ("do", do)):
        _same(q, x, name)
    lse = _lse_like(q, lse, "lse")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, x in (("dq", dq), ("dk", dk), ("dv", dv)):
        _same(q, x, name)
    with torch.cuda.device(q.device):
        code = load().attn_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                       lse.data_ptr(), do.data_ptr(), dq.data_ptr(),
                                       dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                                       _DTYPE_CODES[q.dtype], int(causal), scale,
                                       _stream_handle(stream))
    _check("attn_bwd_noalloc", code)
    return dq, dk, dv


@_on_launch_stream
def attn_bwd_preprocess(o: torch.Tensor, do: torch.Tensor,
                        delta: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """delta = rowsum(do * o) in float32, via libattn.so."""
    B, H, N, d = _shape_of(o, "o")
    _same(o, do, "do")
    delta = _lse_like(o, delta, "delta")
    with torch.cuda.device(o.device):
        code = load().attn_bwd_preprocess(o.data_ptr(), do.data_ptr(), delta.data_ptr(), B, H,
                                          N, d, _DTYPE_CODES[o.dtype], _stream_handle(stream))
    _check("attn_bwd_preprocess", code)
    return delta


@_on_launch_stream
def attn_bwd_dkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lse: torch.Tensor,
                 delta: torch.Tensor, do: torch.Tensor, causal: bool = False,
                 scale: Optional[float] = None, dk: Optional[torch.Tensor] = None,
                 dv: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None
                 ) -> tuple[torch.Tensor, torch.Tensor]:
    """dk, dv from the dK/dV kernel alone (delta from attn_bwd_preprocess)."""
    B, H, N, d = _shape_of(q, "q")
    for name, x in (("k", k), ("v", v), ("do", do)):
        _same(q, x, name)
    lse = _lse_like(q, lse, "lse")
    delta = _lse_like(q, delta, "delta")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    _same(q, dk, "dk")
    _same(q, dv, "dv")
    with torch.cuda.device(q.device):
        code = load().attn_bwd_dkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(),
                                   delta.data_ptr(), do.data_ptr(), dk.data_ptr(),
                                   dv.data_ptr(), B, H, N, d, _DTYPE_CODES[q.dtype],
                                   int(causal), scale, _stream_handle(stream))
    _check("attn_bwd_dkv", code)
    return dk, dv


@_on_launch_stream
def attn_bwd_dq(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lse: torch.Tensor,
                delta: torch.Tensor, do: torch.Tensor, causal: bool = False,
                scale: Optional[float] = None, dq: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """dq from the dQ kernel alone (delta from attn_bwd_preprocess)."""
    B, H, N, d = _shape_of(q, "q")
    for name, x in (("k", k), ("v", v), ("do", do)):
        _same(q, x, name)
    lse = _lse_like(q, lse, "lse")
    delta = _lse_like(q, delta, "delta")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    _same(q, dq, "dq")
    with torch.cuda.device(q.device):
        code = load().attn_bwd_dq(q.data_ptr(), k.data_ptr(), v.data_ptr(), lse.data_ptr(),
                                  delta.data_ptr(), do.data_ptr(), dq.data_ptr(), B, H, N, d,
                                  _DTYPE_CODES[q.dtype], int(causal), scale,
                                  _stream_handle(stream))
    _check("attn_bwd_dq", code)
    return dq


# ---------------------------------------------------------------- host-buffer step
def attn_step_host_scratch_bytes(B: int, H: int, N: int, d: int, chunks: int) -> int:
    return int(load().attn_step_host_scratch_bytes(B, H, N, d, chunks))


@_on_launch_stream
def attn_step_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, do: torch.Tensor,
                   o: torch.Tensor, lse: torch.Tensor, dq: torch.Tensor, dk: torch.Tensor,
                   dv: torch.Tensor, scratch: torch.Tensor, causal: bool = False,
                   scale: Optional[float] = None, chunks: int = 4,
                   stream: Optional[torch.cuda.Stream] = None) -> None:
    """Forward + backward of host (CPU, ideally pinned) tensors through the library,
    copies overlapped with the kernels. Writes o, lse, dq, dk, dv (host tensors); they are
    valid after the stream is synchronised. scratch: a CUDA uint8 tensor of
    attn_step_host_scratch_bytes(B, H, N, d, chunks) bytes."""
    B, H, N, d = q.shape
    for name, x in (("q", q), ("k", k), ("v", v), ("do", do), ("o", o), ("dq", dq), ("dk", dk),
                    ("dv", dv)):
        if x.is_cuda or not x.is_contiguous() or x.shape != q.shape or x.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous host tensor shaped and typed like q")
    if q.dtype not in _DTYPE_CODES:
        raise ValueError("q must be float16 or bfloat16")
    if lse.is_cuda or lse.shape != (B, H, N) or lse.dtype != torch.float32 \
            or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 host tensor [B, H, N]")
    if not scratch.is_cuda or not scratch.is_contiguous():
        raise ValueError("scratch must be a contiguous CUDA tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    nbytes = scratch.numel() * scratch.element_size()
    with torch.cuda.device(scratch.device):
        code = load().attn_step_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                                     o.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                     dk.data_ptr(), dv.data_ptr(), scratch.data_ptr(), nbytes,
                                     B, H, N, d, _DTYPE_CODES[q.dtype], int(causal), scale,
                                     int(chunks), _stream_handle(stream))
    _check("attn_step_host", code)


# ---------------------------------------------------------------- split-KV decode
def attn_decode_splits(B: int, H: int, Nk: int) -> int:
    return int(load().attn_decode_splits(B, H, Nk))


def attn_decode_workspace_bytes(B: int, H: int, d: int, num_splits: int) -> int:
    return int(load().attn_decode_workspace_bytes(B, H, d, num_splits))


def _decode_args(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    B, H, Nq, d = _shape_of(q, "q")
    if Nq != 1:
        raise ValueError("q must hold one query row per (b, h): [B, H, 1, d]")
    Bk, Hk, Nk, dk = _shape_of(k, "k")
    if (Bk, Hk, dk) != (B, H, d) or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k must be [B, H, Nk, d] with q's dtype and device")
    if v.shape != k.shape or v.dtype != k.dtype or v.device != k.device or not v.is_contiguous():
        raise ValueError("v must match k")
    return B, H, Nk, d


def _partials_like(q, B, H, d, splits, partials):
    n = attn_decode_workspace_bytes(B, H, d, splits) // 4
    if partials is None:
        return torch.empty((B, H, splits, d + 4), dtype=torch.float32, device=q.device)
    if partials.dtype != torch.float32 or not partials.is_contiguous() \
            or partials.numel() < n or partials.device != q.device:
        raise ValueError("partials must be a contiguous float32 tensor of "
                         "attn_decode_workspace_bytes / 4 elements on q's device")
    return partials


@_on_launch_stream
def attn_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                scale: Optional[float] = None, num_splits: Optional[int] = None,
                o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                partials: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None
                ) -> tuple[torch.Tensor, torch.Tensor]:
    """Split-KV decode: o = softmax(scale q k^T) v for q [B, H, 1, d], k, v [B, H, Nk, d];
    lse [B, H] float32. Returns (o, lse)."""
    B, H, Nk, d = _decode_args(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    splits = attn_decode_splits(B, H, Nk) if num_splits is None else int(num_splits)
    o = torch.empty_like(q) if o is None else o
    _same(q, o, "o")
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    if lse.shape != (B, H) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H] tensor")
    partials = _partials_like(q, B, H, d, splits, partials)
    with torch.cuda.device(q.device):
        code = load().attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), partials.data_ptr(), B, H, Nk, d,
                                  _DTYPE_CODES[q.dtype], scale, splits, _stream_handle(stream))
    _check("attn_decode", code)
    return o, lse


@_on_launch_stream
def attn_decode_partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        scale: Optional[float] = None, num_splits: int = 1,
                        partials: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """The per-split records [B, H, num_splits, d + 4]: O~ [d], m, l, 2 unused."""
    B, H, Nk, d = _decode_args(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    partials = _partials_like(q, B, H, d, num_splits, partials)
    with torch.cuda.device(q.device):
        code = load().attn_decode_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          partials.data_ptr(), B, H, Nk, d,
                                          _DTYPE_CODES[q.dtype], scale, int(num_splits),
                                          _stream_handle(stream))
    _check("attn_decode_partial", code)
    return partials


@_on_launch_stream
def attn_decode_merge(partials: torch.Tensor, dtype: torch.dtype,
                      o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None
                      ) -> tuple[torch.Tensor, torch.Tensor]:
    """Joins [B, H, S, d + 4] records into o [B, H, 1, d] (dtype) and lse [B, H]."""
    if partials.dim() != 4 or partials.dtype != torch.float32 or not partials.is_contiguous() \
            or not partials.is_cuda:
        raise ValueError("partials must be a contiguous CUDA float32 [B, H, S, d + 4] tensor")
    B, H, S, d4 = partials.shape
    d = d4 - 4
    if o is None:
        o = torch.empty((B, H, 1, d), dtype=dtype, device=partials.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=partials.device)
    _shape_of(o, "o")
    with torch.cuda.device(partials.device):
        code = load().attn_decode_merge(partials.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H,
                                        d, _DTYPE_CODES[o.dtype], S, _stream_handle(stream))
    _check("attn_decode_merge", code)
    return o, lse


def attn_last_kernel_status(stream: Optional[torch.cuda.Stream] = None) -> tuple[int, int]:
    """(status, where): ATTN_ERR_TIMEOUT and the wait's code if a bounded wait ran out."""
    where = ctypes.c_int(0)
    code = load().attn_last_kernel_status(_stream_handle(stream), ctypes.byref(where))
    return int(code), int(where.value)


def status_str(code: int) -> str:
    return load().attn_status_str(code).decode()


# ------------------------------------------------------------------ packed batches

def _packed_of(x: torch.Tensor, name: str) -> tuple[int, int, int]:
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError(f"{name} must be a packed [total, H, d] tensor")
    if not x.is_cuda or not x.is_contiguous() or x.dtype not in _DTYPE_CODES:
        raise ValueError(f"{name} must be a contiguous float16/bfloat16 CUDA tensor")
    return tuple(x.shape)  # type: ignore[return-value]


def _cu_of(cu: torch.Tensor, name: str, device: torch.device) -> torch.Tensor:
    if (not isinstance(cu, torch.Tensor) or cu.dim() != 1 or cu.numel() < 2
            or cu.dtype != torch.int32 or cu.device != device or not cu.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous int32 [B + 1] tensor on q's device")
    return cu


def _host_cu(cu_q_host, cu_k_host, B):
    """Host pointers of the optional CPU copies of cu_seqlens (both or neither)."""
    if cu_q_host is None and cu_k_host is None:
        return None, None
    for name, cu in (("cu_seqlens_q_host", cu_q_host), ("cu_seqlens_k_host", cu_k_host)):
        if (not isinstance(cu, torch.Tensor) or cu.device.type != "cpu" or cu.dtype != torch.int32
                or cu.dim() != 1 or cu.numel() != B + 1 or not cu.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 CPU tensor of B + 1 entries "
                             "(give both host copies or neither)")
    return cu_q_host.data_ptr(), cu_k_host.data_ptr()


def _upload_cpu_cu(q, cu_q, cu_k, cu_q_host, cu_k_host):
    """cu_seqlens given as CPU int32 tensors (both): uploaded to q's device for the kernels,
    and kept as the host copies that order the work unless host copies were given. The
    callers run on their launch stream (_on_launch_stream), so the upload is queued there,
    before the kernels that read it, and its memory belongs to that stream."""
    if (isinstance(cu_q, torch.Tensor) and isinstance(cu_k, torch.Tensor)
            and cu_q.device.type == "cpu" and cu_k.device.type == "cpu"
            and q.device.type == "cuda"):
        if cu_q_host is None and cu_k_host is None:
            cu_q_host, cu_k_host = cu_q.contiguous(), cu_k.contiguous()
        cu_q, cu_k = cu_q.contiguous().to(q.device), cu_k.contiguous().to(q.device)
    return cu_q, cu_k, cu_q_host, cu_k_host


def _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k):
    Tq, H, d = _packed_of(q, "q")
    Tk, Hk, dk = _packed_of(k, "k")
    if (Hk, dk) != (H, d) or k.dtype != q.dtype or k.device != q.device:
        raise ValueError("k must be [total_k, H, d] with q's H, d, dtype and device")
    if v.shape != k.shape or v.dtype != k.dtype or v.device != k.device:
        raise ValueError("v must match k")
    _packed_of(v, "v")
    cu_q = _cu_of(cu_seqlens_q, "cu_seqlens_q", q.device)
    cu_k = _cu_of(cu_seqlens_k, "cu_seqlens_k", q.device)
    if cu_k.numel() != cu_q.numel():
        raise ValueError("cu_seqlens_q and cu_seqlens_k must describe the same batch")
    return Tq, Tk, H, d, cu_q, cu_k, cu_q.numel() - 1


def attn_bwd_varlen_workspace_bytes(H: int, total_q: int) -> int:
    return int(load().attn_bwd_varlen_workspace_bytes(H, total_q))


@_on_launch_stream
def attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                    cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                    max_seqlen_q: int, max_seqlen_k: int, causal: bool = False,
                    scale: Optional[float] = None, o: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None,
                    cu_seqlens_q_host: Optional[torch.Tensor] = None,
                    cu_seqlens_k_host: Optional[torch.Tensor] = None
                    ) -> tuple[torch.Tensor, torch.Tensor]:
    """Forward over sequences packed along the token axis, via libattn.so.

    cu_seqlens_q_host / _k_host: optional CPU int32 copies of the same offsets. They only
    order the kernels' work items (longest first, balanced over the SMs); the results do not
    depend on them. cu_seqlens_q / _k may also be given as CPU int32 tensors: they are then
    uploaded for the kernels and serve as the host copies.

    q [total_q, H, d], k and v [total_k, H, d]; sequence b owns query tokens
    cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens cu_seqlens_k[b] ..
    cu_seqlens_k[b+1]-1 (int32 device tensors of B + 1 entries). max_seqlen_q/_k bound
    every sequence (the caller knows them; reading cu_seqlens here would synchronise).
    Returns o [total_q, H, d] and lse [H, total_q]. Malformed sequences are reported by
    attn_last_kernel_status() as ATTN_ERR_INVALID_ARG."""
    cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host = _upload_cpu_cu(
        q, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host)
    Tq, Tk, H, d, cu_q, cu_k, B = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k)
    hq, hk = _host_cu(cu_seqlens_q_host, cu_seqlens_k_host, B)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if o is None else o
    if o.shape != q.shape or o.dtype != q.dtype or o.device != q.device:
        raise ValueError("o must match q")
    lse = torch.empty(H, Tq, dtype=torch.float32, device=q.device) if lse is None else lse
    if lse.shape != (H, Tq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total_q] tensor")
    with torch.cuda.device(q.device):
        code = load().attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), cu_q.data_ptr(), cu_k.data_ptr(), hq, hk,
                                      B, H, Tq, Tk, int(max_seqlen_q), int(max_seqlen_k), d,
                                      _DTYPE_CODES[q.dtype], int(causal), scale,
                                      _stream_handle(stream))
    _check("attn_fwd_varlen", code)
    return o, lse


@_on_launch_stream
def attn_bwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                    lse: torch.Tensor, do: torch.Tensor, cu_seqlens_q: torch.Tensor,
                    cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
                    causal: bool = False, scale: Optional[float] = None,
                    dq: Optional[torch.Tensor] = None, dk: Optional[torch.Tensor] = None,
                    dv: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None,
                    cu_seqlens_q_host: Optional[torch.Tensor] = None,
                    cu_seqlens_k_host: Optional[torch.Tensor] = None
                    ) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """dq, dk, dv of sum(do * o) for a packed batch (layouts and the optional host copies
    of cu_seqlens as attn_fwd_varlen), via libattn.so; workspace holds D [H, total_q]
    float32."""
    cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host = _upload_cpu_cu(
        q, cu_seqlens_q, cu_seqlens_k, cu_seqlens_q_host, cu_seqlens_k_host)
    Tq, Tk, H, d, cu_q, cu_k, B = _varlen_args(q, k, v, cu_seqlens_q, cu_seqlens_k)
    hq, hk = _host_cu(cu_seqlens_q_host, cu_seqlens_k_host, B)
    for name, x in (("o", o), ("do", do)):
        if x.shape != q.shape or x.dtype != q.dtype or x.device != q.device:
            raise ValueError(f"{name} must match q")
        _packed_of(x, name)
    if lse.shape != (H, Tq) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, total_q] tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    for name, x, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, k)):
        if x.shape != ref.shape or x.dtype != ref.dtype or x.device != ref.device:
            raise ValueError(f"{name} must match {'q' if ref is q else 'k'}")
        _packed_of(x, name)
    if workspace is None:
        workspace = torch.empty(H, Tq, dtype=torch.float32, device=q.device)
    if workspace.numel() * workspace.element_size() < 4 * H * Tq or not workspace.is_contiguous():
        raise ValueError("workspace must hold H * total_q float32 values")
    with torch.cuda.device(q.device):
        code = load().attn_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                      lse.data_ptr(), do.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                      dv.data_ptr(), workspace.data_ptr(), cu_q.data_ptr(),
                                      cu_k.data_ptr(), hq, hk, B, H, Tq, Tk, int(max_seqlen_q),
                                      int(max_seqlen_k), d, _DTYPE_CODES[q.dtype], int(causal),
                                      scale, _stream_handle(stream))
    _check("attn_bwd_varlen", code)
    return dq, dk, dv
