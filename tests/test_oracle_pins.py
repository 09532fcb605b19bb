"""Pins of the fp64 oracle to things other than itself.

Each check ties the oracle to a value the pages print for a worked example, to a
closed form, to brute force on tiny inputs, to finite differences, or to an
independent library routine. ``test_planted_mistakes_are_caught`` plants plausible
mistakes in a copy of the oracle's source (on the CPU) and requires that at least
one pin fails for each.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import scipy.special

import oracle.attention as OA
import oracle.online as OL

HERE = os.path.dirname(os.path.abspath(__file__))
LN = {"0": 0.0, "ln2": math.log(2.0), "ln4": math.log(4.0)}


def _golden(name):
    with open(os.path.join(HERE, "golden", name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------------
# Individual pin checks; each takes an oracle module so that mutants can be checked.
# ----------------------------------------------------------------------------------

def pin_worked_example_a(oa):
    """p5's example run through the definition: weights 1:2:4 give exactly 30."""
    g = _golden("worked_example_a.json")
    k = np.array([[LN[s]] for s in g["scores_scaled"]])
    v = np.array(g["values"])[:, None]
    o, lse = oa.attention_forward(np.array([[1.0]]), k, v, causal=False, scale=1.0)
    assert abs(o[0, 0] - g["output"]) < 1e-12
    assert abs(lse[0] - math.log(7.0)) < 1e-12


def pin_worked_example_b(oa):
    """p4's four-key example: the closed form to 1e-12, the printed value to 2e-3."""
    g = _golden("worked_example_b.json")
    k = np.array(g["scores"])[:, None]
    v = np.array(g["values"])[:, None]
    o, lse = oa.attention_forward(np.array([[1.0]]), k, v, causal=False, scale=1.0)
    e = np.exp(np.array(g["scores"]) - 5.0)
    exact = float((e * np.array(g["values"])).sum() / e.sum())
    assert abs(o[0, 0] - exact) < 1e-12
    assert abs(o[0, 0] - g["output"]) <= g["printed_abs_tolerance"]
    assert abs(lse[0] - (5.0 + math.log(e.sum()))) < 1e-12


def pin_causal_row0_and_n1(oa):
    """Causal row 0 sees key 0 only: O_0 = V_0 and L_0 = S_00. N = 1 likewise."""
    rng = np.random.default_rng(5)
    q, k, v = rng.standard_normal((3, 12, 6))
    scale = 0.37
    o, lse = oa.attention_forward(q, k, v, causal=True, scale=scale)
    assert np.array_equal(o[0], v[0])
    assert abs(lse[0] - scale * float(q[0] @ k[0])) < 1e-14
    o1, l1 = oa.attention_forward(q[:1], k[:1], v[:1], causal=False, scale=scale)
    assert np.array_equal(o1[0], v[0])
    assert abs(l1[0] - scale * float(q[0] @ k[0])) < 1e-14


def pin_uniform_attention(oa):
    """Q = 0 makes every visible score 0: O_i is the mean of the visible V rows and
    L_i = ln(#visible)."""
    rng = np.random.default_rng(6)
    n, d = 17, 5
    k, v = rng.standard_normal((2, n, d))
    q = np.zeros((n, d))
    for causal in (False, True):
        o, lse = oa.attention_forward(q, k, v, causal=causal, scale=0.5)
        for i in range(n):
            cnt = i + 1 if causal else n
            np.testing.assert_allclose(o[i], v[:cnt].mean(axis=0), rtol=0, atol=1e-14)
            assert abs(lse[i] - math.log(cnt)) < 1e-14


def pin_one_hot(oa):
    """One score far above the rest selects that key's value row."""
    n, d = 9, 4
    rng = np.random.default_rng(7)
    v = rng.standard_normal((n, d))
    k = np.zeros((n, d))
    k[6, 0] = 1.0
    q = np.zeros((n, d))
    q[:, 0] = 80.0
    o, lse = oa.attention_forward(q, k, v, causal=False, scale=1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v[6], (n, d)), atol=1e-30 + 1e-12)
    np.testing.assert_allclose(lse, 80.0 + math.log1p((n - 1) * math.exp(-80.0)), atol=1e-12)


def pin_library_softmax(oa):
    """Against scipy's softmax / logsumexp on the explicitly masked score matrix."""
    rng = np.random.default_rng(8)
    n, d = 23, 7
    q, k, v = rng.standard_normal((3, n, d))
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        s = scale * (q @ k.T)
        if causal:
            s[np.triu_indices(n, 1)] = -np.inf
        o, lse = oa.attention_forward(q, k, v, causal=causal, scale=scale)
        np.testing.assert_allclose(lse, scipy.special.logsumexp(s, axis=1), rtol=0, atol=1e-13)
        np.testing.assert_allclose(o, scipy.special.softmax(s, axis=1) @ v, rtol=0, atol=1e-13)


def pin_blocked_recurrence(oa):
    """Naive (definition) versus blocked online recurrence on tiny random inputs,
    every block shape, both masks: 1e-12."""
    for seed in range(12):
        rng = np.random.default_rng(100 + seed)
        n = int(rng.integers(1, 40))
        d = int(rng.integers(1, 9))
        q, k, v = rng.standard_normal((3, n, d)) * rng.uniform(0.5, 3.0)
        scale = float(rng.uniform(0.1, 1.0))
        for causal in (False, True):
            o, lse = oa.attention_forward(q, k, v, causal=causal, scale=scale)
            for bq, bk in ((1, 1), (3, 5), (8, 2), (n, n), (16, 7)):
                ob, lb = OL.blocked_attention(q, k, v, causal, scale, bq, bk)
                np.testing.assert_allclose(ob, o, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(lb, lse, rtol=1e-12, atol=1e-12)


def _fd_check(oa, causal, seed):
    rng = np.random.default_rng(seed)
    n, d = 7, 4
    q, k, v, do = rng.standard_normal((4, n, d))
    scale = 0.6

    def f(qq, kk, vv):
        o, _ = oa.attention_forward(qq, kk, vv, causal=causal, scale=scale)
        return float((do * o).sum())

    g = oa.attention_backward(q, k, v, do, causal=causal, scale=scale)
    h = 1e-6
    for name, idx in (("dq", 0), ("dk", 1), ("dv", 2)):
        base = [q, k, v]
        num = np.zeros((n, d))
        for i in range(n):
            for c in range(d):
                plus = [x.copy() for x in base]
                minus = [x.copy() for x in base]
                plus[idx][i, c] += h
                minus[idx][i, c] -= h
                num[i, c] = (f(*plus) - f(*minus)) / (2 * h)
        err = np.linalg.norm(g[name] - num) / max(1e-30, np.linalg.norm(num))
        assert err <= 1e-6, (name, causal, err)


def pin_finite_differences(oa):
    for causal in (False, True):
        _fd_check(oa, causal, 11 + int(causal))


def pin_delta_two_ways(oa):
    """sum_j P_ij dP_ij equals rowsum(dO_i * O_i) and the stand-alone preprocess."""
    rng = np.random.default_rng(9)
    n, d = 31, 6
    q, k, v, do = rng.standard_normal((4, n, d))
    for causal in (False, True):
        g = oa.attention_backward(q, k, v, do, causal=causal, scale=0.4)
        np.testing.assert_allclose(g["delta"], g["delta_rowsum"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(oa.delta_rowsum(g["o"], do), g["delta_rowsum"], atol=1e-14)
        o, lse = oa.attention_forward(q, k, v, causal=causal, scale=0.4)
        np.testing.assert_allclose(g["o"], o, atol=1e-14)
        np.testing.assert_allclose(g["lse"], lse, atol=1e-14)


def pin_shift_invariance(oa):
    """Adding one vector c to every key shifts row i's scores by scale*q_i.c: O is
    unchanged, L moves by exactly that amount, dQ/dK/dV do not change."""
    rng = np.random.default_rng(10)
    n, d = 13, 5
    q, k, v, do = rng.standard_normal((4, n, d))
    c = rng.standard_normal(d)
    scale = 0.7
    for causal in (False, True):
        o, lse = oa.attention_forward(q, k, v, causal=causal, scale=scale)
        o2, lse2 = oa.attention_forward(q, k + c, v, causal=causal, scale=scale)
        np.testing.assert_allclose(o2, o, atol=1e-12)
        np.testing.assert_allclose(lse2 - lse, scale * (q @ c), atol=1e-12)
        g1 = oa.attention_backward(q, k, v, do, causal=causal, scale=scale)
        g2 = oa.attention_backward(q, k + c, v, do, causal=causal, scale=scale)
        np.testing.assert_allclose(g2["dv"], g1["dv"], atol=1e-12)
        np.testing.assert_allclose(g2["dk"], g1["dk"], atol=1e-12)
        # dQ picks up dS·c per row, and sum_j dS_ij = 0, so dQ is unchanged too.
        np.testing.assert_allclose(g2["dq"], g1["dq"], atol=1e-12)


def pin_causal_future_independence(oa):
    """Changing keys/values after position i leaves O, L and dQ of rows <= i
    bit-for-bit unchanged (masked entries contribute exactly 0)."""
    rng = np.random.default_rng(12)
    n, d = 20, 4
    q, k, v, do = rng.standard_normal((4, n, d))
    i = 9
    k2, v2 = k.copy(), v.copy()
    k2[i + 1:] = rng.standard_normal((n - i - 1, d)) * 5
    v2[i + 1:] = rng.standard_normal((n - i - 1, d)) * 5
    o, lse = oa.attention_forward(q, k, v, causal=True, scale=0.5)
    o2, lse2 = oa.attention_forward(q, k2, v2, causal=True, scale=0.5)
    assert np.array_equal(o[: i + 1], o2[: i + 1])
    assert np.array_equal(lse[: i + 1], lse2[: i + 1])
    g1 = oa.attention_backward(q, k, v, do, causal=True, scale=0.5)
    g2 = oa.attention_backward(q, k2, v2, do, causal=True, scale=0.5)
    assert np.array_equal(g1["dq"][: i + 1], g2["dq"][: i + 1])


def pin_rectangular_is_a_suffix(oa):
    """N_q < N_k (queries last): the rectangular problem equals the last N_q rows of the
    square problem over the same keys; its dK, dV equal the square problem's with dO zero
    on the first N_k - N_q rows, and its dQ equals the square dQ's last rows."""
    rng = np.random.default_rng(23)
    for nk, nq, d, causal in [(9, 4, 3, True), (9, 4, 3, False), (7, 7, 2, True), (12, 1, 4, True)]:
        q = rng.standard_normal((nk, d))
        k = rng.standard_normal((nk, d))
        v = rng.standard_normal((nk, d))
        do = rng.standard_normal((nk, d))
        do[: nk - nq] = 0.0
        sq = oa.attention_backward(q, k, v, do, causal, 0.6)
        rect = oa.attention_backward(q[nk - nq:], k, v, do[nk - nq:], causal, 0.6)
        np.testing.assert_allclose(rect["o"], sq["o"][nk - nq:], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(rect["lse"], sq["lse"][nk - nq:], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(rect["dq"], sq["dq"][nk - nq:], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(rect["dk"], sq["dk"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(rect["dv"], sq["dv"], rtol=1e-10, atol=1e-12)
        o, lse = oa.attention_forward(q[nk - nq:], k, v, causal, 0.6)
        np.testing.assert_allclose(o, sq["o"][nk - nq:], rtol=1e-12, atol=1e-12)
    # the last query row sees every key: it is plain softmax over all of them
    s_last = 0.6 * (k @ q[-1])
    p = scipy.special.softmax(s_last)
    o, lse = oa.attention_forward(q[-1:], k, v, True, 0.6)
    np.testing.assert_allclose(o[0], p @ v, rtol=1e-12, atol=1e-12)


def pin_panels(oa):
    """Whole-row panels change nothing but summation order: 1 row per panel versus
    all rows at once."""
    rng = np.random.default_rng(13)
    n, d = 37, 5
    q, k, v, do = rng.standard_normal((4, n, d))
    for causal in (False, True):
        a = oa.attention_backward(q, k, v, do, causal, 0.3, panel_elems=1)
        b = oa.attention_backward(q, k, v, do, causal, 0.3)
        for key in ("dq", "dk", "dv", "o", "lse", "delta"):
            np.testing.assert_allclose(a[key], b[key], rtol=1e-13, atol=1e-13)


ALL_PINS = [
    pin_worked_example_a, pin_worked_example_b, pin_causal_row0_and_n1,
    pin_uniform_attention, pin_one_hot, pin_library_softmax, pin_blocked_recurrence,
    pin_finite_differences, pin_delta_two_ways, pin_shift_invariance,
    pin_causal_future_independence, pin_panels, pin_rectangular_is_a_suffix,
]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(OA)


# ----------------------------------------------------------------------------------
# The online recurrence itself, against the pages' printed intermediate values.
# ----------------------------------------------------------------------------------

def test_example_a_every_block_split():
    g = _golden("worked_example_a.json")
    s = [LN[x] for x in g["scores_scaled"]]
    for block in (1, 2, 3):
        o, lse, _ = OL.run_row(s, g["values"], block)
        assert abs(o[0] - g["output_every_block_split"]) < 1e-12
        assert abs(lse - math.log(7.0)) < 1e-12


def test_example_a_intermediates():
    g = _golden("worked_example_a.json")
    s = [LN[x] for x in g["scores_scaled"]]
    _, _, trace = OL.run_row(s, g["values"], 2)
    first, second = trace
    assert abs(first.m - LN[g["after_first_block_of_two"]["m"]]) < 1e-15
    assert abs(first.l - g["after_first_block_of_two"]["l"]) < 1e-12
    assert abs(first.u[0] - g["after_first_block_of_two"]["u"]) < 1e-12
    assert abs(OL.rescale_factor(first.m, second.m) - g["after_second_block"]["rescale"]) < 1e-15
    assert abs(second.l - g["after_second_block"]["l"]) < 1e-12
    assert abs(second.u[0] - g["after_second_block"]["u"]) < 1e-12


def test_example_a_negative_control():
    """The page's control that omits the rescale of the old sums gives 26, not 30."""
    g = _golden("worked_example_a.json")
    s = [LN[x] for x in g["scores_scaled"]]
    o_bad, _, _ = OL.run_row(s, g["values"], 2, rescale=False)
    assert abs(o_bad[0] - g["no_rescale_control_output"]) < 1e-12
    o_good, _, _ = OL.run_row(s, g["values"], 2)
    assert abs(o_good[0] - o_bad[0]) > 1.0


def test_example_b_trace():
    g = _golden("worked_example_b.json")
    _, _, trace = OL.run_row(g["scores"], g["values"], 2)
    tol = g["printed_abs_tolerance"]
    for st, key in zip(trace, ("block1", "block2")):
        ref = g[key]
        assert abs(st.m - ref["m"]) < 1e-15
        assert abs(st.l - ref["l"]) <= tol * 1e-1 + 5e-5 * abs(ref["l"])
        assert abs(st.u[0] - ref["o_unnormalised"]) <= tol
    assert abs(OL.rescale_factor(trace[0].m, trace[1].m) - g["block2"]["alpha"]) < 5e-5
    assert OL.rescale_factor(-math.inf, trace[0].m) == g["block1"]["alpha"]
    o, _, _ = OL.run_row(g["scores"], g["values"], 2)
    assert abs(o[0] - g["output"]) <= tol


def test_rescale_factor_p1():
    g = _golden("rescale_factor_p1.json")
    tol = g["printed_digits_abs_tolerance"]
    w1 = math.exp(g["score"] - g["m_chunk1"])
    assert abs(w1 - g["weight_chunk1"]) <= tol["weight_chunk1"]
    w_true = w1 * OL.rescale_factor(g["m_chunk1"], g["m_chunk2"])
    assert abs(w_true - math.exp(g["score"] - g["m_chunk2"])) < 1e-15
    assert abs(w_true - g["weight_true"]) <= tol["weight_true"]


def test_merge_of_partials_is_exact():
    """Split-KV: partial states over disjoint key ranges merge to the full answer."""
    rng = np.random.default_rng(3)
    s = rng.standard_normal(50) * 4
    v = rng.standard_normal((50, 3))
    full, lse_full, _ = OL.run_row(s, v, 50)
    for cut in (1, 17, 49):
        _, _, ta = OL.run_row(s[:cut], v[:cut], 7)
        _, _, tb = OL.run_row(s[cut:], v[cut:], 5)
        o, lse = OL.finish(OL.merge(ta[-1], tb[-1]))
        np.testing.assert_allclose(o, full, atol=1e-12)
        assert abs(lse - lse_full) < 1e-12


# ----------------------------------------------------------------------------------
# Planted mistakes: a copy of the oracle source with one plausible error each.
# ----------------------------------------------------------------------------------

MUTANTS = {
    "dropped_scale_in_dk": ("dk += scale * (ds.T @ q[r0:r1])", "dk += (ds.T @ q[r0:r1])"),
    "dropped_scale_in_dq": ("dq[r0:r1] = scale * (ds @ k)", "dq[r0:r1] = (ds @ k)"),
    "mask_wrong_direction": ("np.where(cols > rows + offset, -np.inf, s)",
                             "np.where(cols < rows + offset, -np.inf, s)"),
    "mask_drops_diagonal": ("np.where(cols > rows + offset, -np.inf, s)",
                            "np.where(cols >= rows + offset, -np.inf, s)"),
    "mask_top_left_aligned": ("offset = k.shape[0] - q.shape[0]", "offset = 0"),
    "mask_offset_sign": ("offset = k.shape[0] - q.shape[0]", "offset = q.shape[0] - k.shape[0]"),
    "lse_in_base2": ("lse[r0:r1] = m + np.log(l)\n    return o, lse",
                     "lse[r0:r1] = m + np.log2(l)\n    return o, lse"),
    "lse_without_max": ("lse[r0:r1] = m + np.log(l)\n    return o, lse",
                        "lse[r0:r1] = np.log(l)\n    return o, lse"),
    "missing_delta_term": ("ds = p * (dp - dlt[:, None])", "ds = p * dp"),
    "transposed_dv": ("dv += p.T @ do_p", "dv += p @ do_p if p.shape[0] == p.shape[1] else p.T @ do_p"),
    "unnormalised_p": ("return e / l[:, None], m, l", "return e, m, l"),
    "sign_error_in_ds": ("ds = p * (dp - dlt[:, None])", "ds = p * (dlt[:, None] - dp)"),
    "dk_uses_k": ("dk += scale * (ds.T @ q[r0:r1])", "dk += scale * (ds.T @ k[r0:r1])"),
}


def _mutant(old, new):
    src = open(OA.__file__).read()
    assert src.count(old) == 1, f"planted-mistake target not found once: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
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
