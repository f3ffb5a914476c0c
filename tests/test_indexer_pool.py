"""Pins for the indexer pooling oracle ("One guard, 110x off the verify step",
section "The same bug, one layer over"): windows of four pooled by their mean,
completed windows kept and the tail recomputed for any number of new tokens,
the four guards, and the top-k window selection.  CPU only."""

import itertools

import numpy as np
import pytest

from oracle import indexer_pool as P


def _keys(rng, T, d=8):
    return rng.standard_normal((T, d))


def test_pool_matches_reshaped_sum():
    # written another way: zero-pad to whole windows, sum each window with a
    # reshape, divide by how many real tokens it holds
    rng = np.random.default_rng(0)
    for T in (1, 3, 4, 5, 8, 13, 64, 67):
        k = _keys(rng, T)
        W = -(-T // 4)
        padded = np.zeros((4 * W, k.shape[1]))
        padded[:T] = k
        counts = np.minimum(4, T - 4 * np.arange(W))
        want = padded.reshape(W, 4, -1).sum(axis=1) / counts[:, None]
        np.testing.assert_allclose(P.pool_all(k, T), want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("S", [2, 3, 4, 8])
@pytest.mark.parametrize("T0", [12, 13, 14, 15, 16])   # aligned and misaligned lengths
def test_wide_step_equals_one_at_a_time(S, T0):
    rng = np.random.default_rng(S * 100 + T0)
    keys = _keys(rng, T0 + S)
    start, _ = P.pool_step(None, keys, T0, T0)            # the pool before the step
    wide, inc = P.pool_step(start, keys, T0 + S, S)
    assert inc
    one = start
    for t in range(T0 + 1, T0 + S + 1):
        one, inc1 = P.pool_step(one, keys, t, 1)
        assert inc1
    assert wide["length"] == one["length"] == T0 + S
    assert np.array_equal(wide["pooled"], one["pooled"])
    assert np.array_equal(wide["pooled"], P.pool_all(keys, T0 + S))


def test_incremental_step_reads_only_the_tail():
    # windows completed before the step come from the pool, not the keys
    rng = np.random.default_rng(5)
    keys = _keys(rng, 30)
    state, _ = P.pool_step(None, keys, 26, 26)
    changed = keys.copy()
    changed[:24] += 100.0                 # windows 0..5 were complete at 26
    new, inc = P.pool_step(state, changed, 30, 4)
    assert inc
    assert np.array_equal(new["pooled"][:6], state["pooled"][:6])
    assert np.array_equal(new["pooled"][6:], P.pool_all(changed, 30)[6:])


@pytest.mark.parametrize("guard", ["no_pool", "padded", "batch", "length"])
def test_each_guard_forces_a_full_recompute(guard):
    rng = np.random.default_rng(7)
    keys = _keys(rng, 40)
    state, _ = P.pool_step(None, keys, 35, 35)
    kw = dict(T=37, S=2)
    if guard == "no_pool":
        state = None
    elif guard == "padded":
        kw["padded"] = True
    elif guard == "batch":
        kw["batch"] = 2
    else:
        kw = dict(T=36, S=2)              # the pool remembers 35, the cache held 34
    new, inc = P.pool_step(state, keys, **kw)
    assert not inc
    assert np.array_equal(new["pooled"], P.pool_all(keys, kw["T"]))


def test_rejection_trim_does_not_carry_stale_windows():
    # pool at 20 tokens; a rejection trims the cache to 17 and two new tokens
    # arrive (T = 19): window 4 (positions 16..19) must come from the new keys
    rng = np.random.default_rng(9)
    old = _keys(rng, 20)
    state, _ = P.pool_step(None, old, 20, 20)
    new_keys = old.copy()
    new_keys[17:19] = rng.standard_normal((2, old.shape[1]))
    new, inc = P.pool_step(state, new_keys, 19, 2)
    assert not inc
    assert np.array_equal(new["pooled"], P.pool_all(new_keys, 19))
    assert not np.allclose(new["pooled"][4], state["pooled"][4])


def test_planted_missing_length_guard_is_caught(monkeypatch):
    real = P.pool_step

    def no_length_guard(state, keys, T, S, padded=False, batch=1):
        if state is not None:
            state = dict(state, length=T - S)   # pretends the pool matches
        return real(state, keys, T, S, padded, batch)

    monkeypatch.setattr(P, "pool_step", no_length_guard)
    with pytest.raises(AssertionError):
        test_rejection_trim_does_not_carry_stale_windows()


def _brute_topk(q, pooled, p, k):
    vis = p // 4 + 1
    best, best_key = None, None
    for combo in itertools.combinations(range(vis), min(k, vis)):
        score = sum(float(pooled[w] @ q) for w in combo)
        key = (score, [-w for w in combo])
        if best_key is None or key > best_key:
            best, best_key = combo, key
    return sorted(best)


def test_select_matches_brute_force_with_causal_limit():
    rng = np.random.default_rng(11)
    for T, S, k in ((13, 3, 2), (16, 4, 3), (9, 2, 5), (30, 1, 4)):
        keys = _keys(rng, T, d=6)
        pooled = P.pool_all(keys, T)
        q = rng.standard_normal((S, 6))
        wins, pos = P.select_topk(q, pooled, T, S, k)
        for s in range(S):
            p = T - S + s
            want = _brute_topk(q[s], pooled, p, k)
            got = [int(w) for w in wins[s] if w >= 0]
            assert got == want
            flat = [4 * w + i for w in want for i in range(4) if 4 * w + i <= p]
            assert list(pos[s, :len(flat)]) == flat
            assert np.all(pos[s, len(flat):] == -1)
            assert all(0 <= x <= p for x in flat)


def test_select_ties_go_to_the_lower_window():
    pooled = np.ones((6, 2))
    q = np.array([[1.0, 0.0]])
    wins, _ = P.select_topk(q, pooled, 24, 1, 3)
    assert list(wins[0]) == [0, 1, 2]


def test_budget_of_512_windows_is_2048_positions():
    rng = np.random.default_rng(13)
    T = 4096
    pooled = P.pool_all(_keys(rng, T, d=4), T)
    _, pos = P.select_topk(rng.standard_normal((1, 4)), pooled, T, 1, 512)
    assert pos.shape == (1, 2048) and np.all(pos >= 0)
    assert len(set(pos[0].tolist())) == 2048
