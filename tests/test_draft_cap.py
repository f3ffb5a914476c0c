"""Draft-cap selection ("Draft caps and calibration", the cost model "in
formula form, for a cap C"): the oracle against the closed form, a worked
example and the page's qualitative statements; the library's
mla_select_draft_cap against the oracle.  CPU only."""

import math

import numpy as np
import pytest

from oracle import draft_cap as D
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    yield


@pytest.mark.parametrize("p", [0.0, 0.1, 0.5, 0.84, 0.999, 1.0])
def test_accepted_is_the_geometric_series(p):
    # 1 + p + ... + p^C = (1 - p^(C+1)) / (1 - p), and C + 1 at p = 1
    for C in range(0, 20):
        want = C + 1 if p == 1.0 else (1 - p ** (C + 1)) / (1 - p)
        assert math.isclose(D.accepted(p, C), want, rel_tol=1e-12, abs_tol=1e-15)


def test_worked_example_by_hand():
    # p = 0.8, verify(w) = 1, 1.5, 2, 2.5, 3 steps, drafter 0.1 step:
    # speedup = 1, 1.8/1.6 = 1.125, 2.44/2.1 = 1.1619, 2.952/2.6 = 1.1354,
    # 3.3616/3.1 = 1.0844 -> cap 2
    cap, s = D.select_draft_cap(0.8, [1, 1.5, 2, 2.5, 3], [0.1], 8)
    assert cap == 2
    np.testing.assert_allclose(s, [1, 1.125, 2.44 / 2.1, 2.952 / 2.6, 3.3616 / 3.1], rtol=1e-12)


def test_flat_verify_curve_drafts_a_lot():
    # "verifying 8 rows costs about the same as 1, so the answer is 'draft a
    # lot'": with a flat curve, once drafting pays at all, the largest
    # measured cap wins (accepted(C) only grows with C)
    for p in (0.3, 0.7, 0.95):
        cap, _ = D.select_draft_cap(p, [1.0] * 8, [0.2], 16)
        assert cap == 7
    # and where it never pays (1 + p + ... < 1 + drafter), plain decoding
    cap, _ = D.select_draft_cap(0.05, [1.0] * 8, [0.2], 16)
    assert cap == 0


def test_no_acceptance_means_no_drafting():
    cap, s = D.select_draft_cap(0.0, [1, 1.1, 1.2], [0.05], 4)
    assert cap == 0 and s[0] == 1.0


def test_drafter_cost_moves_the_cap_the_provable_way():
    # With a drafter cost per drafted token, d*C, a costlier drafter never
    # raises the cap: accepted(C)/C falls with C, so once the smaller of two
    # caps wins at some d it wins at every larger d.  With a fixed cost per
    # round it is the other way round among the caps that draft at all (C >= 1;
    # plain decoding, C = 0, pays no drafter): the fixed cost is spread over
    # more committed tokens, and the best drafting cap never falls as d grows.
    rng = np.random.default_rng(3)
    for _ in range(50):
        curve = list(np.cumsum(np.r_[1.0, rng.uniform(0.0, 0.6, 15)]))
        p = float(rng.uniform(0.3, 0.95))
        ds = np.linspace(0, 3, 13)
        per_token = [D.select_draft_cap(p, curve, [d * C for C in range(16)], 15)[0] for d in ds]
        def best_drafting(d):
            sp = D.select_draft_cap(p, curve, [d], 15)[1]
            return 1 + int(np.argmax(sp[1:]))
        per_round = [best_drafting(d) for d in ds]
        assert all(a >= b for a, b in zip(per_token, per_token[1:])), per_token
        assert all(a <= b for a, b in zip(per_round, per_round[1:])), per_round


def test_planted_off_by_one_in_accepted_is_caught(monkeypatch):
    monkeypatch.setattr(D, "accepted", lambda p, C: sum(p ** i for i in range(C)))
    with pytest.raises(AssertionError):
        test_worked_example_by_hand()


def test_library_matches_oracle():
    rng = np.random.default_rng(11)
    for _ in range(300):
        n = int(rng.integers(1, 20))
        curve = list(np.cumsum(np.r_[rng.uniform(1, 50), rng.uniform(0, 30, n - 1)]))
        per_cap = bool(rng.integers(0, 2))
        dr = list(rng.uniform(0, 20, n + 2)) if per_cap else [float(rng.uniform(0, 20))]
        p = float(rng.uniform(0, 1))
        mc = int(rng.integers(0, 24))
        want, ws = D.select_draft_cap(p, curve, dr, mc)
        got, gs = B.mla_select_draft_cap(p, curve, dr, mc)
        assert got == want
        assert gs == ws           # same arithmetic in the same order: bit for bit


@pytest.mark.parametrize("p,curve,dr,mc", [
    (1.5, [1, 2], [0.1], 4),        # p outside [0, 1]
    (-0.1, [1, 2], [0.1], 4),
    (0.5, [1, 0], [0.1], 4),        # a verify cost of zero
    (0.5, [1, 2], [-1.0], 4),       # a negative drafter cost
    (0.5, [1, 2], [0.1], -1),       # negative max cap
])
def test_library_rejects_bad_arguments(p, curve, dr, mc):
    with pytest.raises(B.MlaError):
        B.mla_select_draft_cap(p, curve, dr, mc)
