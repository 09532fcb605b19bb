"""Pins of the packed variable-length oracle (oracle/varlen.py) to things other than itself.

* Brute force on tiny inputs: a plain Python loop over every (token, head) with math.exp,
  no max shift and no matrices, summing over exactly the keys of the token's own
  sequence that the bottom-right causal mask leaves visible.
* The pages' worked example ("FlashAttention·FA4·FP4", section 온라인 softmax가 블록 사이의
  값을 어떻게 이어 주나; tests/golden/worked_example_a.json) packed as the middle one of
  three sequences: its query still gives exactly 30 and L = ln 7, whatever the other
  sequences hold.
* Isolation: changing the tokens of other sequences leaves a sequence's O, L and
  gradients bit-for-bit unchanged.
* Central finite differences of sum(dO * O) over the whole packed batch.
* One sequence (B = 1): each head equals oracle.attention on that head's rows (the
  special case that reduces to the dense oracle, itself pinned in test_oracle_pins.py).

``test_planted_mistakes_are_caught`` plants plausible mistakes in a copy of the oracle's
source (on the CPU) and requires that at least one pin fails for each.
"""
import json
import math
import os
import types

import numpy as np
import pytest

import oracle.attention as OA
import oracle.varlen as OV

HERE = os.path.dirname(os.path.abspath(__file__))

# (cu_q, cu_k, causal): empty sequences, n_k > n_q, n_k < n_q without the mask.
LAYOUTS = [
    ([0, 3, 3, 7, 8], [0, 5, 6, 10, 12], True),
    ([0, 3, 3, 7, 8], [0, 5, 6, 10, 12], False),
    ([0, 4, 5, 9], [0, 2, 3, 5], False),
    ([0, 6], [0, 6], True),
    ([0, 1, 2, 3], [0, 1, 2, 3], True),
]


def _rand(cu_q, cu_k, H=2, d=3, seed=0):
    rng = np.random.default_rng(seed)
    tq, tk = cu_q[-1], cu_k[-1]
    return (rng.standard_normal((tq, H, d)), rng.standard_normal((tk, H, d)),
            rng.standard_normal((tk, H, d)), rng.standard_normal((tq, H, d)))


def _brute(q, k, v, cu_q, cu_k, causal, scale):
    tq, H, d = q.shape
    o = np.zeros((tq, H, v.shape[2]))
    lse = np.zeros((H, tq))
    for b in range(len(cu_q) - 1):
        nq, nk = cu_q[b + 1] - cu_q[b], cu_k[b + 1] - cu_k[b]
        for i in range(nq):
            t = cu_q[b] + i
            for h in range(H):
                num = [0.0] * v.shape[2]
                den = 0.0
                for j in range(nk):
                    if causal and j > i + (nk - nq):
                        continue
                    u = cu_k[b] + j
                    w = math.exp(scale * sum(q[t, h, c] * k[u, h, c] for c in range(d)))
                    den += w
                    for c in range(v.shape[2]):
                        num[c] += w * v[u, h, c]
                o[t, h] = [x / den for x in num]
                lse[h, t] = math.log(den)
    return o, lse


def pin_brute_force(ov):
    for n, (cu_q, cu_k, causal) in enumerate(LAYOUTS):
        q, k, v, _ = _rand(cu_q, cu_k, seed=n)
        o, lse = ov.varlen_forward(q, k, v, cu_q, cu_k, causal, 0.7)
        o_b, lse_b = _brute(q, k, v, cu_q, cu_k, causal, 0.7)
        assert np.abs(o - o_b).max() < 1e-12, (cu_q, cu_k, causal)
        assert np.abs(lse - lse_b).max() < 1e-12, (cu_q, cu_k, causal)


def pin_worked_example_packed(ov):
    with open(os.path.join(HERE, "golden", "worked_example_a.json")) as f:
        g = json.load(f)
    ln = {"0": 0.0, "ln2": math.log(2.0), "ln4": math.log(4.0)}
    rng = np.random.default_rng(5)
    cu_q, cu_k = [0, 2, 3, 5], [0, 4, 7, 9]
    q = rng.standard_normal((5, 1, 1))
    k = rng.standard_normal((9, 1, 1))
    v = rng.standard_normal((9, 1, 1))
    q[2, 0, 0] = 1.0
    k[4:7, 0, 0] = [ln[s] for s in g["scores_scaled"]]
    v[4:7, 0, 0] = g["values"]
    for causal in (False, True):  # one query, three keys: the mask hides nothing
        o, lse = ov.varlen_forward(q, k, v, cu_q, cu_k, causal, 1.0)
        assert abs(o[2, 0, 0] - g["output"]) < 1e-12
        assert abs(lse[0, 2] - math.log(7.0)) < 1e-12


def pin_isolation(ov):
    cu_q, cu_k, causal = [0, 3, 3, 7, 8], [0, 5, 6, 10, 12], True
    q, k, v, do = _rand(cu_q, cu_k, seed=3)
    ref = ov.varlen_backward(q, k, v, do, cu_q, cu_k, causal, 0.5)
    q2, k2, v2, do2 = (x.copy() for x in (q, k, v, do))
    b = 2  # change every sequence but b
    for x, cu in ((q2, cu_q), (k2, cu_k), (v2, cu_k), (do2, cu_q)):
        x[:cu[b]] += 1.5
        x[cu[b + 1]:] -= 2.5
    got = ov.varlen_backward(q2, k2, v2, do2, cu_q, cu_k, causal, 0.5)
    for name, cu in (("o", cu_q), ("dq", cu_q), ("dk", cu_k), ("dv", cu_k)):
        assert np.array_equal(got[name][cu[b]:cu[b + 1]], ref[name][cu[b]:cu[b + 1]]), name
        assert not np.array_equal(got[name][:cu[b]], ref[name][:cu[b]]), name
    assert np.array_equal(got["lse"][:, cu_q[b]:cu_q[b + 1]], ref["lse"][:, cu_q[b]:cu_q[b + 1]])


def pin_finite_differences(ov):
    for cu_q, cu_k, causal in LAYOUTS[:3]:
        q, k, v, do = _rand(cu_q, cu_k, d=2, seed=7)
        g = ov.varlen_backward(q, k, v, do, cu_q, cu_k, causal, 0.9)

        def f(q_, k_, v_):
            return float((ov.varlen_forward(q_, k_, v_, cu_q, cu_k, causal, 0.9)[0] * do).sum())

        eps = 1e-6
        for name, x in (("dq", q), ("dk", k), ("dv", v)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += eps
                xm[idx] -= eps
                args_p = [q, k, v]
                args_m = [q, k, v]
                pos = {"dq": 0, "dk": 1, "dv": 2}[name]
                args_p[pos], args_m[pos] = xp, xm
                num[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
            err = np.linalg.norm(g[name] - num) / max(np.linalg.norm(num), 1e-300)
            assert err < 1e-6, (cu_q, cu_k, causal, name, err)
        d_ref = (do * g["o"]).sum(axis=2).T
        assert np.abs(g["delta"] - d_ref).max() < 1e-12


def pin_single_sequence(ov):
    cu = [0, 9]
    q, k, v, do = _rand(cu, cu, H=3, d=4, seed=11)
    for causal in (False, True):
        o, lse = ov.varlen_forward(q, k, v, cu, cu, causal, 0.6)
        for h in range(3):
            o_d, l_d = OA.attention_forward(q[:, h], k[:, h], v[:, h], causal, 0.6)
            assert np.abs(o[:, h] - o_d).max() < 1e-13
            assert np.abs(lse[h] - l_d).max() < 1e-13


ALL_PINS = [pin_brute_force, pin_worked_example_packed, pin_isolation, pin_finite_differences,
            pin_single_sequence]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(OV)


def test_malformed_layouts_are_rejected():
    q, k, v, _ = _rand([0, 4], [0, 4])
    for cu_q, cu_k, causal in (([0, 5], [0, 4], False), ([1, 4], [0, 4], False),
                               ([0, 4], [0, 3], True), ([0, 2, 4], [0, 5, 4], False)):
        with pytest.raises(ValueError):
            OV.varlen_forward(q, k, v, cu_q, cu_k, causal, 1.0)


MUTANTS = {
    # keys taken from the query boundaries
    "keys_from_cu_q": ("k0, k1 = _bounds(cu_k, b)\n        _check_pair(q1 - q0, k1 - k0, causal)\n"
                       "        if q1 == q0:\n            continue\n",
                       "k0, k1 = _bounds(cu_q, b)\n        _check_pair(q1 - q0, k1 - k0, causal)\n"
                       "        if q1 == q0:\n            continue\n"),
    # a query sees the keys of every earlier sequence too (no segmentation)
    "keys_from_start": ("OA.attention_forward(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h]",
                        "OA.attention_forward(q[q0:q1, h], k[:k1, h], v[:k1, h]"),
    # one key past the sequence end
    "key_end_off_by_one": ("ob, lb = OA.attention_forward(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h]",
                           "ob, lb = OA.attention_forward(q[q0:q1, h], k[k0:k1 + 1, h], "
                           "v[k0:k1 + 1, h]"),
    # last sequence dropped
    "last_sequence_dropped": ("    o = np.zeros((q.shape[0], H, v.shape[2]))\n"
                              "    lse = np.zeros((H, q.shape[0]))\n"
                              "    for b in range(cu_q.size - 1):",
                              "    o = np.zeros((q.shape[0], H, v.shape[2]))\n"
                              "    lse = np.zeros((H, q.shape[0]))\n"
                              "    for b in range(cu_q.size - 2):"),
    # dk written at the query positions
    "dk_at_query_rows": ('out["dk"][k0:k1, h] = r["dk"]', 'out["dk"][q0:q0 + (k1 - k0), h] = r["dk"]'),
    # lse of head h written into head 0
    "lse_head_index": ("lse[h, q0:q1] = lb", "lse[0, q0:q1] = lb"),
}


def _mutant(old, new):
    src = open(OV.__file__).read()
    assert src.count(old) == 1, f"planted-mistake target not found once: {old!r}"
    mod = types.ModuleType("oracle_varlen_mutant")
    exec(compile(src.replace(old, new), "oracle_varlen_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
