"""Pins of the split-KV decode oracle (oracle/decode.py) to things other than itself.

* The pages' worked example ("FlashAttention·FA4·FP4", section 온라인 softmax가 블록 사이의
  값을 어떻게 이어 주나; tests/golden/worked_example_a.json): the partial state of the
  first two keys and the merge with the third are printed there, and every split of the
  three keys gives 30.
* The plain definition: the merge of the partial states of any split equals softmax
  attention over all keys (oracle.attention.attention_forward, itself pinned in
  test_oracle_pins.py), to 1e-12.
* Order independence of the merge, neutral empty parts, and the split rule's coverage.

``test_planted_mistakes_are_caught`` plants plausible mistakes in a copy of the decode
oracle's source (on the CPU) and requires that one of the pins fails for each.
"""
import itertools
import json
import math
import os
import types

import numpy as np
import pytest

import oracle.attention as OA
import oracle.decode as OD

HERE = os.path.dirname(os.path.abspath(__file__))
LN = {"0": 0.0, "ln2": math.log(2.0), "ln4": math.log(4.0)}


def _golden(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


def _example():
    g = _golden("worked_example_a.json")
    k = np.array([[LN[s]] for s in g["scores_scaled"]])
    v = np.array(g["values"])[:, None]
    return g, np.array([1.0]), k, v


def pin_example_states(od):
    """First two keys: m = ln 2, l = 1.5, u = 25; joined with the third key: m = ln 4,
    l = 1.75, u = 52.5; O = 30 (the page's numbers)."""
    g, q, k, v = _example()
    m, l, u = od.partial_state(q, k, v, 1.0, 0, 2)
    first = g["after_first_block_of_two"]
    assert abs(m - LN[first["m"]]) < 1e-12
    assert abs(l - first["l"]) < 1e-12 and abs(u[0] - first["u"]) < 1e-12
    m2, l2, u2 = od.merge_states([(m, l, u), od.partial_state(q, k, v, 1.0, 2, 3)])
    second = g["after_second_block"]
    assert abs(m2 - LN[second["m"]]) < 1e-12
    assert abs(l2 - second["l"]) < 1e-12 and abs(u2[0] - second["u"]) < 1e-12
    o, lse = od.finish(m2, l2, u2)
    assert abs(o[0] - g["output"]) < 1e-12
    assert abs(lse - math.log(7.0)) < 1e-12  # e^0 + e^ln2 + e^ln4 = 7


def pin_example_every_split(od):
    """Every cut of the three keys into contiguous parts merges to 30."""
    g, q, k, v = _example()
    for cuts in itertools.product([False, True], repeat=2):
        edges = [0] + [i + 1 for i, c in enumerate(cuts) if c] + [3]
        parts = [od.partial_state(q, k, v, 1.0, a, b) for a, b in zip(edges, edges[1:])]
        o, lse = od.finish(*od.merge_states(parts))
        assert abs(o[0] - g["output_every_block_split"]) < 1e-12


def pin_definition(od):
    """Merged partials == softmax attention over all keys, for many splits."""
    rng = np.random.default_rng(7)
    for nk, d, scale in [(1, 4, 0.5), (63, 8, 0.35), (64, 8, 1.0), (65, 16, 0.25),
                         (300, 64, 0.125), (1000, 8, 0.7)]:
        q = rng.standard_normal(d)
        k = rng.standard_normal((nk, d)) * 2.0
        v = rng.standard_normal((nk, d))
        ref_o, ref_l = OA.attention_forward(q[None, :], k, v, False, scale)
        for splits in (1, 2, 3, 7, 16, 100):
            o, lse, parts = od.decode(q, k, v, scale, splits)
            assert len(parts) == splits
            np.testing.assert_allclose(o, ref_o[0], rtol=1e-12, atol=1e-12)
            assert abs(lse - ref_l[0]) < 1e-12


def pin_order_and_neutral(od):
    """Any order of the parts, and extra empty parts, give the same merged state."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal(8)
    k = rng.standard_normal((500, 8)) * 3.0
    v = rng.standard_normal((500, 8))
    parts = [od.partial_state(q, k, v, 0.4, a, b)
             for a, b in [(0, 64), (64, 200), (200, 256), (256, 500)]]
    m0, l0, u0 = od.merge_states(parts)
    neutral = (-math.inf, 0.0, np.zeros(8))
    for perm in itertools.permutations(range(4)):
        m, l, u = od.merge_states([parts[i] for i in perm] + [neutral])
        assert abs(m - m0) < 1e-12 and abs(l / l0 - 1) < 1e-12
        np.testing.assert_allclose(u, u0, rtol=1e-12, atol=1e-12)
    m, l, u = od.merge_states([neutral, neutral] + parts)
    assert abs(m - m0) < 1e-12 and abs(l / l0 - 1) < 1e-12


def pin_split_rule(od):
    """The splits cover [0, Nk) once, in order, in multiples of 64 keys."""
    for nk in (1, 63, 64, 65, 1000, 4096, 32769):
        for splits in (1, 2, 5, 8, 64, 600):
            b = od.split_bounds(nk, splits)
            assert len(b) == splits and b[0][0] == 0 and b[-1][1] == nk
            for (a0, a1), (c0, c1) in zip(b, b[1:]):
                assert a1 == c0 and a0 <= a1
            c = od.split_length(nk, splits)
            assert c % 64 == 0 and c >= -(-nk // splits)
            assert all(k1 - k0 in (0, c) or k1 == nk for k0, k1 in b)


PINS = [pin_example_states, pin_example_every_split, pin_definition,
        pin_order_and_neutral, pin_split_rule]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_decode_oracle_pin(pin):
    pin(OD)


MUTANTS = {
    "merge_l_without_rescale": ("l = a * l + b * l_p", "l = l + l_p"),
    "merge_u_without_rescale": ("u = a * u + b * u_p", "u = u + u_p"),
    "merge_weight_swapped": ("b = math.exp(m_p - m_new)", "b = math.exp(m - m_new)"),
    "lse_without_max": ("return u / l, m + math.log(l)", "return u / l, math.log(l)"),
    "partial_without_shift": ("e = np.exp(s - m)", "e = np.exp(s)"),
    "partial_without_scale": ("s = scale * (k[k0:k1] @ q)", "s = (k[k0:k1] @ q)"),
    "split_not_aligned": ("return SPLIT_ALIGN * (-(-per // SPLIT_ALIGN))", "return per"),
}


def _mutant(old, new):
    with open(OD.__file__) as f:
        src = f.read()
    assert old in src, old
    mod = types.ModuleType("decode_mutant")
    exec(compile(src.replace(old, new), "decode_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError, FloatingPointError, ZeroDivisionError):
            failed += 1
    assert failed > 0, f"mutant {name} passed every pin"
