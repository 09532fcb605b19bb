"""Packed variable-length batches (attn_fwd_varlen / attn_bwd_varlen through the binding)
versus the fp64 oracle (oracle/varlen.py), element by element on every sequence and head,
with the tolerances of tests/parity.py; plus bit-for-bit identities with the dense
entry points, isolation of sequences, untouched tokens outside every sequence, and
malformed cu_seqlens reported through the status word.
"""
import numpy as np
import pytest
import torch

import oracle.attention as OA
import oracle.varlen as OV
from exact_attention_tcgen05_gb300 import binding
from exact_attention_tcgen05_gb300 import inputs as I

from parity import GRAD_TOL, LSE_TOL, o_error, record, rel_fro

pytestmark = pytest.mark.gpu

CASES = [
    # H, d, dtype, causal, query lengths, key lengths (None: same)
    (2, 128, "bf16", True, (1, 130, 257, 64, 700), None),
    (2, 64, "fp16", False, (300, 17, 513), None),
    (1, 128, "fp16", True, (129, 128, 383), (400, 128, 1000)),    # more keys: bottom-right
    (2, 64, "bf16", False, (200, 64, 1), (90, 300, 5)),           # fewer keys, no mask
    (2, 128, "bf16", True, (0, 77, 0, 256), (0, 77, 40, 300)),    # empty query sequences
    (3, 64, "bf16", True, (1000,), None),                         # one sequence
    (2, 64, "bf16", False, (1100, 40, 700), None),  # long enough for K, V in tensor memory
    (2, 96, "bf16", True, (300, 129, 64), (310, 200, 64)),  # a head dim of 96
    # head dims above 128: the 256-column kernels
    (2, 256, "bf16", True, (1, 130, 257, 64, 700), None),
    (1, 192, "fp16", True, (129, 128, 383), (400, 128, 1000)),
    (2, 256, "bf16", True, (0, 77, 0, 256), (0, 77, 40, 300)),   # keys without queries
    (2, 256, "fp16", False, (200, 64, 1), (90, 300, 5)),
]


def _tensors(w):
    q, do = (I.make_varlen_tensor(w, t).cuda() for t in ("q", "do"))
    k, v = (I.make_varlen_tensor(w, t).cuda() for t in ("k", "v"))
    cu_q = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    return q, k, v, do, cu_q, cu_k


def _run(w, q, k, v, do, cu_q, cu_k):
    o, lse = binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, w.max_q, w.max_k, causal=w.causal,
                                     scale=w.scale)
    dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, w.max_q, w.max_k,
                                         causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def _f64(x):
    return x.detach().cpu().double().numpy()


@pytest.mark.parametrize("case", CASES, ids=lambda c: "H{}d{}_{}_{}_q{}_k{}".format(
    c[0], c[1], c[2], "causal" if c[3] else "full", "-".join(map(str, c[4])),
    "-".join(map(str, c[5] or c[4]))))
def test_packed_matches_oracle(case):
    H, d, dtype, causal, lq, lk = case
    w = I.varlen(H, d, dtype, causal, seed=70 + sum(lq), seqlens_q=lq, seqlens_k=lk)
    q, k, v, do, cu_q, cu_k = _tensors(w)
    o, lse, dq, dk, dv = _run(w, q, k, v, do, cu_q, cu_k)
    assert binding.attn_last_kernel_status() == (0, 0)
    ref = OV.varlen_backward(_f64(q), _f64(k), _f64(v), _f64(do), w.cu_q, w.cu_k, causal,
                             w.scale)
    og, lg = _f64(o), lse.cpu().double().numpy()
    dqg, dkg, dvg = _f64(dq), _f64(dk), _f64(dv)
    for b in range(w.B):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        k0, k1 = w.cu_k[b], w.cu_k[b + 1]
        for h in range(H):
            where = f"sequence {b} head {h}"
            if q1 > q0:
                r = o_error(og[q0:q1, h], ref["o"][q0:q1, h], w.torch_dtype)
                assert r["o_excess"] <= 0, f"{where}: O error {r['o_max']:.3e}"
                assert np.abs(lg[h, q0:q1] - ref["lse"][h, q0:q1]).max() <= LSE_TOL, where
                assert rel_fro(dqg[q0:q1, h], ref["dq"][q0:q1, h]) <= GRAD_TOL, where
            if k1 > k0:
                if q1 == q0:  # keys no query sees: exactly zero
                    assert not dkg[k0:k1, h].any() and not dvg[k0:k1, h].any(), where
                else:
                    assert rel_fro(dkg[k0:k1, h], ref["dk"][k0:k1, h]) <= GRAD_TOL, where
                    assert rel_fro(dvg[k0:k1, h], ref["dv"][k0:k1, h]) <= GRAD_TOL, where


@pytest.mark.parametrize("d,causal", [(128, True), (64, False), (256, True), (200, False)])
def test_equal_lengths_equal_the_dense_call_bit_for_bit(d, causal):
    """B sequences of one length N, packed, give exactly the bits of attn_fwd/attn_bwd on
    the [B, H, N, d] tensors (the same tiles in the same order)."""
    B, H, N = 3, 2, 300
    w = I.varlen(H, d, "bf16", causal, seed=5, seqlens_q=(N,) * B)
    q, k, v, do, cu_q, cu_k = _tensors(w)
    o, lse, dq, dk, dv = _run(w, q, k, v, do, cu_q, cu_k)

    def dense(x):  # [B*N, H, d] -> [B, H, N, d]
        return x.view(B, N, H, d).permute(0, 2, 1, 3).contiguous()

    od, lsed = binding.attn_fwd(dense(q), dense(k), dense(v), causal=causal, scale=w.scale)
    dqd, dkd, dvd = binding.attn_bwd(dense(q), dense(k), dense(v), od, lsed, dense(do),
                                     causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dense(o), od)
    assert torch.equal(lse.view(H, B, N).permute(1, 0, 2), lsed)
    for got, want in ((dq, dqd), (dk, dkd), (dv, dvd)):
        assert torch.equal(dense(got), want)


def test_other_sequences_do_not_leak():
    w = I.varlen(2, 128, "bf16", True, seed=8, seqlens_q=(200, 333, 150),
                 seqlens_k=(260, 333, 400))
    q, k, v, do, cu_q, cu_k = _tensors(w)
    ref = _run(w, q, k, v, do, cu_q, cu_k)
    b = 1
    for x, cu in ((q, w.cu_q), (k, w.cu_k), (v, w.cu_k), (do, w.cu_q)):
        x[:cu[b]] *= -2
        x[cu[b + 1]:] += 3
    got = _run(w, q, k, v, do, cu_q, cu_k)
    q0, q1, k0, k1 = w.cu_q[b], w.cu_q[b + 1], w.cu_k[b], w.cu_k[b + 1]
    assert torch.equal(got[0][q0:q1], ref[0][q0:q1])
    assert torch.equal(got[1][:, q0:q1], ref[1][:, q0:q1])
    assert torch.equal(got[2][q0:q1], ref[2][q0:q1])
    assert torch.equal(got[3][k0:k1], ref[3][k0:k1])
    assert torch.equal(got[4][k0:k1], ref[4][k0:k1])
    assert not torch.equal(got[0][:q0], ref[0][:q0])


def test_tokens_outside_every_sequence_are_not_written():
    w = I.varlen(2, 64, "fp16", False, seed=9, seqlens_q=(100, 50), seqlens_k=(80, 60))
    q, k, v, do, _, _ = _tensors(w)
    # The boundaries cover only the first 120 query and 110 key tokens.
    cu_q = torch.tensor([0, 70, 120], dtype=torch.int32, device="cuda")
    cu_k = torch.tensor([0, 60, 110], dtype=torch.int32, device="cuda")
    o = torch.full_like(q, 7.0)
    lse = torch.full((2, q.shape[0]), 7.0, device="cuda")
    binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, 70, 60, o=o, lse=lse)
    dk = torch.full_like(k, 7.0)
    binding.attn_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, 70, 60, dk=dk)
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    assert bool((o[120:] == 7).all()) and bool((lse[:, 120:] == 7).all())
    assert bool((dk[110:] == 7).all()) and not bool((dk[:110] == 7).any())


@pytest.mark.parametrize("cu_q,cu_k,max_q,causal", [
    ([0, 50, 40, 100], [0, 50, 90, 100], 60, False),   # decreasing boundary
    ([0, 50, 100, 100], [0, 50, 100, 100], 40, False),  # a sequence longer than max_seqlen
    ([0, 50, 100, 100], [0, 50, 60, 100], 50, True),    # causal with fewer keys
    ([0, 50, 100, 100], [0, 50, 50, 100], 50, False),   # queries without keys
    ([0, 50, 100, 130], [0, 50, 100, 100], 50, False),  # past the end of q
])
def test_malformed_boundaries_are_reported(cu_q, cu_k, max_q, causal):
    H, d = 2, 64
    q = torch.randn(100, H, d, device="cuda", dtype=torch.bfloat16)
    k = torch.randn(100, H, d, device="cuda", dtype=torch.bfloat16)
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    binding.attn_fwd_varlen(q, k, k, cq, ck, max_q, 60, causal=causal)
    torch.cuda.synchronize()
    code, where = binding.attn_last_kernel_status()
    assert code == 1 and where == 0x7E
    # the context is still usable and the status word was cleared
    w = I.varlen(H, d, "bf16", False, seed=1, seqlens_q=(30, 70))
    q2, k2, v2, do2, cu_q2, cu_k2 = _tensors(w)
    _run(w, q2, k2, v2, do2, cu_q2, cu_k2)
    assert binding.attn_last_kernel_status() == (0, 0)


def test_bench_batch_sampled_against_the_oracle():
    """The packed benchmark batch (16384 tokens, 32 heads, d = 128, causal) at full size,
    in the launch configuration the benchmark times; the shortest and the longest
    sequence are checked against the oracle on two heads each."""
    w = I.VARLEN_BENCH
    q, k, v, do, cu_q, cu_k = _tensors(w)
    o, lse, dq, dk, dv = _run(w, q, k, v, do, cu_q, cu_k)
    assert binding.attn_last_kernel_status() == (0, 0)
    lengths = list(w.seqlens_q)
    for b in (lengths.index(min(lengths)), lengths.index(max(lengths))):
        q0, q1 = w.cu_q[b], w.cu_q[b + 1]
        for h in (0, w.H - 1):
            ref = OA.attention_backward(_f64(q[q0:q1, h]), _f64(k[q0:q1, h]), _f64(v[q0:q1, h]),
                                        _f64(do[q0:q1, h]), True, w.scale)
            r = o_error(_f64(o[q0:q1, h]), ref["o"], w.torch_dtype)
            r["lse_max"] = float(np.abs(lse[h, q0:q1].cpu().double().numpy() - ref["lse"]).max())
            for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
                r[name] = rel_fro(_f64(got[q0:q1, h]), ref[name])
            record(f"{w.name} (sequence {b})", r)
            assert r["o_excess"] <= 0, (b, h, r["o_max"])
            assert r["lse_max"] <= LSE_TOL
            for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
                assert rel_fro(_f64(got[q0:q1, h]), ref[name]) <= GRAD_TOL, (b, h, name)


@pytest.mark.parametrize("causal,d,lq,lk", [
    (True, 128, (700, 1, 1500, 129, 2048, 300, 999, 64), None),
    (False, 64, (200, 1800, 64, 1, 900, 1300), (250, 1800, 100, 7, 1000, 1300)),
])
def test_host_lengths_only_order_the_work(causal, d, lq, lk):
    """With host copies of cu_seqlens the persistent kernels walk their items in a greedy
    longest-first order (more items than SMs here); the results are those of the call
    without them, bit for bit - also when the host copies are wrong, since every item slot
    is computed from the device copies whatever the host copies say."""
    w = I.varlen(16, d, "bf16", causal, seed=90 + d, seqlens_q=lq, seqlens_k=lk)
    q, k, v, do, cu_q, cu_k = _tensors(w)

    def run(hq, hk):
        o, lse = binding.attn_fwd_varlen(q, k, v, cu_q, cu_k, w.max_q, w.max_k, causal=causal,
                                         scale=w.scale, cu_seqlens_q_host=hq,
                                         cu_seqlens_k_host=hk)
        dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, cu_q, cu_k, w.max_q, w.max_k,
                                             causal=causal, scale=w.scale,
                                             cu_seqlens_q_host=hq, cu_seqlens_k_host=hk)
        torch.cuda.synchronize()
        assert binding.attn_last_kernel_status() == (0, 0)
        return o, lse, dq, dk, dv

    base = run(None, None)
    right = run(torch.tensor(w.cu_q, dtype=torch.int32), torch.tensor(w.cu_k, dtype=torch.int32))
    # wrong host lengths: the sequences' lengths in reverse order
    rev_q = np.concatenate([[0], np.cumsum(list(reversed(w.seqlens_q)))]).astype(np.int32)
    rev_k = np.concatenate([[0], np.cumsum(list(reversed(w.seqlens_k)))]).astype(np.int32)
    wrong = run(torch.from_numpy(rev_q), torch.from_numpy(rev_k))
    for name, a, b, c in zip(("O", "LSE", "dQ", "dK", "dV"), base, right, wrong):
        assert torch.equal(a, b), f"{name}: host lengths changed the result"
        assert torch.equal(a, c), f"{name}: wrong host lengths changed the result"


def test_cpu_cu_seqlens_are_uploaded_and_order_the_work():
    """cu_seqlens given as CPU tensors: the binding uploads them for the kernels and uses
    them as the host copies; the results are those of device cu_seqlens, bit for bit."""
    w = I.varlen(8, 128, "bf16", True, seed=123, seqlens_q=(900, 33, 1500, 257, 640))
    q, k, v, do, cu_q, cu_k = _tensors(w)
    ref = _run(w, q, k, v, do, cu_q, cu_k)
    got = _run(w, q, k, v, do, cu_q.cpu(), cu_k.cpu())
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), ref, got):
        assert torch.equal(a, b), name


def test_cpu_cu_seqlens_on_a_side_stream():
    """The same call on a stream other than torch's current one: the binding uploads the
    CPU cu_seqlens and allocates the outputs and workspace on that stream, so they are in
    place before its kernels run and no allocation on the current stream can take their
    memory meanwhile (small int32 buffers filled with -1 are allocated there while the
    side stream runs). Bit-identical to the call on the default stream."""
    w = I.varlen(8, 128, "bf16", True, seed=124, seqlens_q=(700, 45, 1300, 129, 512))
    q, k, v, do, cu_q, cu_k = _tensors(w)
    ref = _run(w, q, k, v, do, cu_q, cu_k)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    hq, hk = cu_q.cpu(), cu_k.cpu()
    o, lse = binding.attn_fwd_varlen(q, k, v, hq, hk, w.max_q, w.max_k, causal=w.causal,
                                     scale=w.scale, stream=side)
    dq, dk, dv = binding.attn_bwd_varlen(q, k, v, o, lse, do, hq, hk, w.max_q, w.max_k,
                                         causal=w.causal, scale=w.scale, stream=side)
    junk = [torch.full((64,), -1, dtype=torch.int32, device="cuda") for _ in range(16)]
    torch.cuda.synchronize()
    assert binding.attn_last_kernel_status() == (0, 0)
    for name, a, b in zip(("O", "LSE", "dQ", "dK", "dV"), ref, (o, lse, dq, dk, dv)):
        assert torch.equal(a, b), name
    del junk
