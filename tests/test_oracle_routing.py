"""Pins for the oracle's router (top-k, combine weights) and sort-free placement.

Checks against things other than the oracle itself:
* brute force over every k-subset of experts;
* hand-worked examples in tests/golden/routing_examples.json;
* exp_rn compared with numpy's fp64 exp;
* the population-count formula for the rank, against the oracle's counting loop;
* invariants: every pair is placed exactly once, no tile holds more than 8 rows,
  and tiles = ceil(count / 8).
"""
import itertools
import json
import os

import numpy as np

import oracle
import synth
from oracle.routing import TILE_ROWS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ulp32(x):
    x = np.abs(np.asarray(x, dtype=np.float32))
    return np.spacing(x).astype(np.float64)


def test_exp_rn_accuracy_against_fp64_exp():
    x = np.concatenate([
        np.linspace(-40.0, 0.0, 200001, dtype=np.float32),
        -np.exp2(np.linspace(-30, 5, 2001)).astype(np.float32),
        np.array([0.0, -0.0, -1e-8, -0.34657359, -0.34657362, -0.6931472, -87.0, -103.0], dtype=np.float32),
    ])
    got = oracle.exp_rn(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    err_ulp = np.abs(got - ref) / ulp32(ref.astype(np.float32))
    assert err_ulp.max() <= 2.0, err_ulp.max()
    assert oracle.exp_rn(np.float32(0.0)) == 1.0


def test_exp_rn_subnormal_range_and_underflow():
    x = np.linspace(-103.9, -87.5, 5001, dtype=np.float32)
    got = oracle.exp_rn(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    # absolute error within 2 ulp of the smallest normal spacing (subnormal step 2^-149)
    assert np.all(np.abs(got - ref) <= np.maximum(2 * ulp32(ref.astype(np.float32)), 2.0 ** -148))
    assert oracle.exp_rn(np.float32(-200.0)) == 0.0


def test_topk_matches_brute_force_subsets():
    rng = np.random.default_rng(11)
    for E, k in [(8, 1), (8, 2), (8, 3), (10, 4), (6, 6)]:
        logits = rng.standard_normal((50, E)).astype(np.float32)
        ids = oracle.topk_ids(logits, k)
        for t in range(50):
            best = max(itertools.combinations(range(E), k), key=lambda c: sum(float(logits[t, i]) for i in c))
            assert set(ids[t]) == set(best)
            vals = logits[t, ids[t]]
            assert np.all(np.diff(vals) < 0)  # descending, distinct here


def test_topk_tie_break_lower_id():
    logits = np.array([[1.0, 2.0, 2.0, 2.0, 0.0]], dtype=np.float32)
    np.testing.assert_array_equal(oracle.topk_ids(logits, 2), [[1, 2]])
    np.testing.assert_array_equal(oracle.topk_ids(logits, 4), [[1, 2, 3, 0]])


def test_router_hand_worked_examples():
    d = json.load(open(os.path.join(GOLDEN, "routing_examples.json")))
    for c in d["topk_cases"]:
        lg = np.array(c["logits"], dtype=np.float32)
        ids = oracle.topk_ids(lg, c["k"])
        np.testing.assert_array_equal(ids, c["ids"])
        w = oracle.softmax_topk_weights(lg, ids)
        exp_w = np.array(c["weights"])
        if c.get("exact"):
            np.testing.assert_array_equal(w.astype(np.float64), exp_w)
        else:
            assert np.all(np.abs(w - exp_w) <= 4 * ulp32(exp_w.astype(np.float32))), (w, exp_w)
    for c in d["placement_cases"]:
        p = oracle.placement(np.array(c["ids"]), c["E"])
        np.testing.assert_array_equal(p["counts"], c["counts"])
        np.testing.assert_array_equal(p["bitmap"], np.array(c["bitmap"], dtype=np.uint32))
        np.testing.assert_array_equal(p["slot_tile"], c["slot_tile"])
        np.testing.assert_array_equal(p["slot_row"], c["slot_row"])


def test_weights_invariants_and_closed_form():
    lg = synth.router_logits(5, 64, 256, 8, "zipf")
    ids = oracle.topk_ids(lg, 8)
    w = oracle.softmax_topk_weights(lg, ids)
    assert np.all(w > 0)
    assert np.all(np.diff(w, axis=1) <= 0)                       # follows the rank order
    assert np.all(np.abs(w.astype(np.float64).sum(axis=1) - 1.0) <= 1e-6)
    # against the closed form in fp64
    sel = np.take_along_axis(lg, ids.astype(np.int64), 1).astype(np.float64)
    ref = np.exp(sel - sel[:, :1])
    ref /= ref.sum(axis=1, keepdims=True)
    assert np.all(np.abs(w - ref) <= 8 * ulp32(ref.astype(np.float32)))


def _popc(x):
    return bin(int(x)).count("1")


def test_placement_popcount_formula_and_invariants():
    for T, E, k, routing in [(6, 8, 2, "uniform"), (40, 8, 2, "uniform"), (96, 256, 8, "zipf"), (70, 16, 3, "zipf")]:
        lg = synth.router_logits(9, T, E, k, routing)
        ids = oracle.topk_ids(lg, k)
        p = oracle.placement(ids, E)
        words = (T + 31) // 32
        seen = set()
        for t in range(T):
            for j in range(k):
                e = int(ids[t, j])
                # rank by population count of bitmap bits below t (a different formula)
                w_, b_ = divmod(t, 32)
                rank = sum(_popc(p["bitmap"][e, i]) for i in range(w_)) + _popc(int(p["bitmap"][e, w_]) & ((1 << b_) - 1))
                assert p["slot_e"][t, j] == e
                assert p["slot_tile"][t, j] * TILE_ROWS + p["slot_row"][t, j] == rank
                assert 0 <= p["slot_row"][t, j] < TILE_ROWS
                key = (e, int(p["slot_tile"][t, j]), int(p["slot_row"][t, j]))
                assert key not in seen
                seen.add(key)
                assert p["rows_of"][e][rank] == t * k + j
        assert len(seen) == T * k
        assert p["counts"].sum() == T * k
        np.testing.assert_array_equal(p["counts"], [sum(_popc(x) for x in p["bitmap"][e]) for e in range(E)])
        np.testing.assert_array_equal(p["tiles"], (p["counts"] + 7) // 8)
        for e in range(E):
            toks = [int(q) // k for q in p["rows_of"][e]]
            assert toks == sorted(toks)                             # ascending token order
            for j in range(int(p["tiles"][e]) - 1):                 # all but the last tile are full
                assert sum(1 for (ee, tt, _) in seen if ee == e and tt == j) == TILE_ROWS
        assert p["bitmap"].shape == (E, words)


def test_exp_rn_constants_are_correctly_rounded():
    """The binary32 constants of exp_rn are the correctly rounded values of
    log2(e), ln2 - ln2_hi and 1/i!, computed here from 60-digit references."""
    sympy = __import__("pytest").importorskip("sympy")
    from fractions import Fraction

    from oracle import routing as R

    def rn32(fr):
        f = np.float32(float(fr))
        cands = [np.nextafter(f, np.float32(0)), f, np.nextafter(f, np.float32(np.inf))]
        return min(cands, key=lambda c: abs(Fraction(float(c)) - fr))

    fact = [1, 1, 2, 6, 24, 120, 720, 5040, 40320]
    for i, f in enumerate(fact):
        assert R._INV_FACT[i] == rn32(Fraction(1, f))
    assert R._LOG2E == rn32(Fraction(str(sympy.N(1 / sympy.log(2), 60))))
    hi = Fraction(45426, 65536)
    assert Fraction(float(R._LN2_HI)) == hi
    assert R._LN2_LO == rn32(Fraction(str(sympy.N(sympy.log(2), 60))) - hi)
