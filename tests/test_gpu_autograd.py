"""The torch.autograd.Function wrappers: forward and backward through autograd give exactly
the bits of the direct binding calls (dense, N_q != N_k, packed batches)."""
import pytest
import torch

from exact_attention_tcgen05_gb300 import autograd, binding
from exact_attention_tcgen05_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Nq,Nk,d,causal", [(300, 300, 128, True), (128, 700, 64, True),
                                            (257, 100, 128, False)])
def test_dense_autograd_matches_binding(Nq, Nk, d, causal):
    wq = I.custom(2, 2, Nq, d, "bf16", causal, seed=Nq)
    wk = I.custom(2, 2, Nk, d, "bf16", causal, seed=Nk + 1)
    q, do = (I.make_tensor(wq, t).cuda() for t in ("q", "do"))
    k, v = (I.make_tensor(wk, t).cuda() for t in ("k", "v"))
    o_ref, lse = binding.attn_fwd(q, k, v, causal=causal)
    dq_ref, dk_ref, dv_ref = binding.attn_bwd(q, k, v, o_ref, lse, do, causal=causal)
    qg, kg, vg = (x.clone().requires_grad_() for x in (q, k, v))
    o = autograd.attention(qg, kg, vg, causal=causal)
    o.backward(do)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    assert torch.equal(qg.grad, dq_ref) and torch.equal(kg.grad, dk_ref)
    assert torch.equal(vg.grad, dv_ref)


def test_packed_autograd_matches_binding():
    w = I.varlen(2, 64, "fp16", True, seed=4, seqlens_q=(300, 1, 520),
                 seqlens_k=(300, 64, 700))
    q, do = (I.make_varlen_tensor(w, t).cuda() for t in ("q", "do"))
    k, v = (I.make_varlen_tensor(w, t).cuda() for t in ("k", "v"))
    cq = torch.tensor(w.cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(w.cu_k, dtype=torch.int32, device="cuda")
    o_ref, lse = binding.attn_fwd_varlen(q, k, v, cq, ck, w.max_q, w.max_k, causal=True)
    ref = binding.attn_bwd_varlen(q, k, v, o_ref, lse, do, cq, ck, w.max_q, w.max_k,
                                  causal=True)
    qg, kg, vg = (x.clone().requires_grad_() for x in (q, k, v))
    o = autograd.attention_varlen(qg, kg, vg, cq, ck, w.max_q, w.max_k, causal=True)
    o.backward(do)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    for got, want in zip((qg.grad, kg.grad, vg.grad), ref):
        assert torch.equal(got, want)
    # with the host copies of cu_seqlens (they only order the work): the same bits
    qg2, kg2, vg2 = (x.clone().requires_grad_() for x in (q, k, v))
    o2 = autograd.attention_varlen(qg2, kg2, vg2, cq, ck, w.max_q, w.max_k, causal=True,
                                   cu_seqlens_q_host=cq.cpu(), cu_seqlens_k_host=ck.cpu())
    o2.backward(do)
    torch.cuda.synchronize()
    assert torch.equal(o2, o_ref)
    for got, want in zip((qg2.grad, kg2.grad, vg2.grad), ref):
        assert torch.equal(got, want)


def test_calls_from_a_thread_without_cuda_context():
    """A host thread that has made no CUDA call has no current context; the C ABI's own
    driver call (tensor-map encoding) must still work there, as it must in the autograd
    engine's worker threads. The results equal the main thread's bit for bit."""
    import threading
    w = I.custom(2, 2, 300, 128, "bf16", True, seed=5)
    q, k, v, do = (I.make_tensor(w, t).cuda() for t in ("q", "k", "v", "do"))
    o_ref, lse_ref = binding.attn_fwd(q, k, v, causal=True)
    grads_ref = binding.attn_bwd(q, k, v, o_ref, lse_ref, do, causal=True)
    torch.cuda.synchronize()
    out, errors = {}, []

    def worker():
        try:
            o, lse = binding.attn_fwd(q, k, v, causal=True)
            out["r"] = (o, lse) + tuple(binding.attn_bwd(q, k, v, o, lse, do, causal=True))
            torch.cuda.synchronize()
        except Exception as e:  # reported below, on the test's thread
            errors.append(e)

    t = threading.Thread(target=worker)
    t.start()
    t.join(timeout=120)
    assert not errors, errors
    for a, b in zip(out["r"], (o_ref, lse_ref) + tuple(grads_ref)):
        assert torch.equal(a, b)
