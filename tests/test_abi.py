"""The C ABI without a GPU: the library builds, exports every function include/attn.h
declares, and rejects bad arguments on the host before making any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_tcgen05_gb300 import binding
    from exact_attention_tcgen05_gb300 import build as B
    B.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes",
                     "attn_bwd_preprocess", "attn_bwd_dkv", "attn_bwd_dq", "attn_status_str",
                     "attn_last_kernel_status"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    from exact_attention_tcgen05_gb300 import build as B
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        getattr(lib, name)


def test_binding_covers_the_header():
    from exact_attention_tcgen05_gb300 import binding
    assert sorted(binding.SIGNATURES) == declared_functions()


def test_status_strings(lib):
    assert lib.attn_status_str(0) == b"ATTN_OK"
    assert lib.attn_status_str(4) == b"ATTN_ERR_TIMEOUT"
    assert lib.attn_status_str(77) == b"ATTN_ERR_UNKNOWN"


def test_workspace_bytes(lib):
    assert lib.attn_bwd_workspace_bytes(4, 32, 4096) == 4 * 4 * 32 * 4096
    assert lib.attn_bwd_workspace_bytes(0, 1, 1) == 0
    assert lib.attn_bwd_workspace_bytes(1, 1, -5) == 0


# Fake, 16-byte aligned, non-overlapping "device" addresses: validation must reject the
# call before any of them is dereferenced or passed to CUDA.
MB = 1 << 20
Q, K, V, O, L, DO, DQ, DK, DV, WS = (0x10000000 + i * 64 * MB for i in range(10))


def fwd(lib, q=Q, k=K, v=V, o=O, lse=L, B=1, H=1, N=256, d=128, dt=1, causal=0, scale=0.1):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, dt, causal, scale, None)


def bwd(lib, dq=DQ, ws=WS, q=Q, B=1, H=1, N=256, d=128, dt=1, scale=0.1):
    return lib.attn_bwd(q, K, V, O, L, DO, dq, DK, DV, ws, B, H, N, d, dt, 0, scale, None)


INVALID, UNSUPPORTED = 1, 2


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), INVALID), (dict(o=0), INVALID), (dict(lse=L + 4), INVALID),
    (dict(k=K + 2), INVALID), (dict(B=0), INVALID), (dict(H=-1), INVALID),
    (dict(N=0), INVALID), (dict(N=(1 << 20) + 1), INVALID), (dict(B=300, H=300), INVALID),
    (dict(d=100), UNSUPPORTED), (dict(d=264), UNSUPPORTED), (dict(d=132), UNSUPPORTED),
    (dict(d=4), UNSUPPORTED), (dict(dt=2), INVALID),
    (dict(scale=0.0), INVALID), (dict(scale=-1.0), INVALID), (dict(scale=float("nan")), INVALID),
    (dict(scale=float("inf")), INVALID), (dict(o=Q), INVALID), (dict(o=K + 16), INVALID),
    (dict(lse=O + 1024), INVALID),
])
def test_fwd_rejects_bad_arguments(lib, kw, code):
    assert fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(dq=0), INVALID), (dict(ws=0), INVALID), (dict(dq=DK), INVALID), (dict(ws=Q), INVALID),
    (dict(dq=O + 32), INVALID), (dict(d=132), UNSUPPORTED), (dict(scale=0.0), INVALID),
    (dict(d=264), UNSUPPORTED),
    (dict(ws=WS + 8), INVALID),
])
def test_bwd_rejects_bad_arguments(lib, kw, code):
    assert bwd(lib, **kw) == code


def fwd_qk(lib, Nq=256, Nk=1024, causal=1, o=O, d=128):
    return lib.attn_fwd_qk(Q, K, V, o, L, 1, 2, Nq, Nk, d, 1, causal, 0.1, None)


def bwd_qk(lib, Nq=256, Nk=1024, causal=1, dk=DK):
    return lib.attn_bwd_qk(Q, K, V, O, L, DO, DQ, dk, DV, WS, 1, 2, Nq, Nk, 128, 1, causal,
                           0.1, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=1024, Nk=256), INVALID),            # causal needs N_k >= N_q
    (dict(Nk=0), INVALID), (dict(Nq=0), INVALID), (dict(Nk=(1 << 20) + 1), INVALID),
    (dict(d=64, o=K + 64 * 1024 * 2 * 2 - 16), INVALID),   # o overlaps the tail of k
    (dict(d=84), UNSUPPORTED),
])
def test_fwd_qk_rejects_bad_arguments(lib, kw, code):
    assert fwd_qk(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=1024, Nk=256), INVALID), (dict(Nk=-3), INVALID),
    (dict(dk=DV + 1024 * 128 * 2 * 2 - 32), INVALID),      # dk overlaps the tail of dv
])
def test_bwd_qk_rejects_bad_arguments(lib, kw, code):
    assert bwd_qk(lib, **kw) == code


CUQ, CUK = 0x10000000 + 10 * 64 * MB, 0x10000000 + 10 * 64 * MB + 4096


# Host copies of cu_seqlens (read on the host only to order work): B = 4 sequences.
HOST_CU = (ctypes.c_int * 5)(0, 250, 500, 750, 1000)
HOST_CU_ADDR = ctypes.addressof(HOST_CU)


def fwd_varlen(lib, q=Q, o=O, cu_q=CUQ, cu_k=CUK, B=4, H=2, Tq=1000, Tk=1200, mq=400, mk=500,
               d=128, dt=1, scale=0.1, hq=None, hk=None):
    return lib.attn_fwd_varlen(q, K, V, o, L, cu_q, cu_k, hq, hk, B, H, Tq, Tk, mq, mk, d, dt, 1,
                               scale, None)


def bwd_varlen(lib, dk=DK, ws=WS, cu_q=CUQ, Tq=1000, mq=400, hq=None, hk=None):
    return lib.attn_bwd_varlen(Q, K, V, O, L, DO, DQ, dk, DV, ws, cu_q, CUK, hq, hk, 4, 2, Tq,
                               1200, mq, 500, 128, 1, 1, 0.1, None)


@pytest.mark.parametrize("kw,code", [
    (dict(cu_q=0), INVALID), (dict(cu_k=0), INVALID), (dict(cu_q=CUQ + 2), INVALID),
    (dict(B=0), INVALID), (dict(Tq=0), INVALID), (dict(mq=0), INVALID),
    (dict(mq=1001), INVALID),                    # longer than the whole packed tensor
    (dict(mk=(1 << 20) + 1, Tk=1 << 21), INVALID), (dict(d=84), UNSUPPORTED),
    (dict(scale=0.0), INVALID), (dict(q=Q + 8), INVALID),
    (dict(o=Q + 1000 * 2 * 128 * 2 - 16), INVALID),  # o overlaps the tail of q
    (dict(o=CUQ - 16), INVALID),                    # o overlaps cu_seqlens_q
    (dict(hq=HOST_CU_ADDR), INVALID), (dict(hk=HOST_CU_ADDR), INVALID),  # one host copy alone
])
def test_fwd_varlen_rejects_bad_arguments(lib, kw, code):
    assert fwd_varlen(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), INVALID), (dict(dk=DV + 16), INVALID), (dict(ws=CUK), INVALID),
    (dict(mq=2000), INVALID), (dict(hq=HOST_CU_ADDR), INVALID),
])
def test_bwd_varlen_rejects_bad_arguments(lib, kw, code):
    assert bwd_varlen(lib, **kw) == code


def test_varlen_workspace_bytes(lib):
    assert lib.attn_bwd_varlen_workspace_bytes(32, 16384) == 4 * 32 * 16384
    assert lib.attn_bwd_varlen_workspace_bytes(0, 5) == 0


def test_stage_entry_points_reject_bad_arguments(lib):
    dkv = lambda dk=DK, dv=DV, d=128, lse=L: lib.attn_bwd_dkv(Q, K, V, lse, WS, DO, dk, dv, 1, 1,
                                                              256, d, 1, 1, 0.1, None)
    assert dkv(dk=DV) == INVALID
    assert dkv(dk=Q) == INVALID
    assert dkv(lse=0) == INVALID
    assert dkv(d=84) == UNSUPPORTED
    dq = lambda out=DQ, scale=0.1: lib.attn_bwd_dq(Q, K, V, L, WS, DO, out, 1, 1, 256, 64, 0, 0,
                                                   scale, None)
    assert dq(out=WS) == INVALID
    assert dq(out=DQ + 4) == INVALID
    assert dq(scale=-2.0) == INVALID


def decode(lib, q=Q, k=K, v=V, o=O, lse=L, part=WS, B=1, H=1, N=256, d=128, dt=1, scale=0.1,
           splits=4):
    return lib.attn_decode(q, k, v, o, lse, part, B, H, N, d, dt, scale, splits, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), INVALID), (dict(part=0), INVALID), (dict(part=WS + 8), INVALID),
    (dict(splits=0), INVALID), (dict(splits=65536), INVALID), (dict(N=0), INVALID),
    (dict(d=96), UNSUPPORTED), (dict(dt=3), INVALID), (dict(scale=0.0), INVALID),
    (dict(o=K), INVALID), (dict(lse=V + 16), INVALID), (dict(part=Q), INVALID),
    (dict(B=300, H=300), INVALID),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert decode(lib, **kw) == code


def test_step_host_rejects_bad_arguments(lib):
    need = lib.attn_step_host_scratch_bytes(1, 2, 256, 128, 2)
    assert need > 0 and lib.attn_step_host_scratch_bytes(1, 2, 256, 100, 2) == 0
    assert lib.attn_step_host_scratch_bytes(1, 2, 256, 96, 2) > 0  # any multiple of 8 <= 256
    assert lib.attn_step_host_scratch_bytes(1, 2, 256, 256, 2) > 0
    assert lib.attn_step_host_scratch_bytes(1, 2, 256, 264, 2) == 0

    def call(scratch=WS, nbytes=need, chunks=2, d=128, scale=0.1, q=Q):
        return lib.attn_step_host(q, K, V, DO, O, L, DQ, DK, DV, scratch, nbytes, 1, 2, 256, d,
                                  1, 0, scale, chunks, None)
    assert call(scratch=0) == INVALID
    assert call(nbytes=need - 1) == INVALID
    assert call(chunks=0) == INVALID
    assert call(d=100) == UNSUPPORTED
    assert call(scale=-1.0) == INVALID
    assert call(q=Q + 8) == INVALID


def test_decode_sizes(lib):
    assert lib.attn_decode_workspace_bytes(2, 3, 128, 5) == 4 * 2 * 3 * 5 * 132
    assert lib.attn_decode_workspace_bytes(2, 3, 96, 5) == 0
    assert lib.attn_decode_workspace_bytes(0, 3, 64, 5) == 0
    assert lib.attn_decode_splits(0, 1, 100) == 0
    # merge validation happens before any CUDA call too
    assert lib.attn_decode_merge(0, O, L, 1, 1, 128, 1, 4, None) == INVALID
    assert lib.attn_decode_merge(WS, O, L, 1, 1, 128, 1, 0, None) == INVALID
    assert lib.attn_decode_merge(WS, WS, L, 1, 1, 128, 1, 4, None) == INVALID


def test_preprocess_rejects_bad_arguments(lib):
    assert lib.attn_bwd_preprocess(O, DO, 0, 1, 1, 16, 64, 0, None) == INVALID
    assert lib.attn_bwd_preprocess(O, DO, O, 1, 1, 16, 64, 0, None) == INVALID
    assert lib.attn_bwd_preprocess(O, DO, WS, 1, 1, 16, 44, 0, None) == UNSUPPORTED


def test_binding_refuses_cpu_tensors():
    import torch
    from exact_attention_tcgen05_gb300 import binding
    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.attn_fwd(x, x, x)


def test_product_path_has_no_oracle_or_fallback():
    """The package never imports the oracle and has no CPU implementation."""
    pkg = os.path.join(ROOT, "exact_attention_tcgen05_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            src = open(os.path.join(pkg, fn)).read()
            assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), fn
            code = re.sub(r'""".*?"""', "", src, flags=re.S)
            code = re.sub(r"#.*", "", code)
            for banned in ("softmax(", "scaled_dot_product", ".exp(", "matmul(", " @ "):
                assert banned not in code, (fn, banned)
