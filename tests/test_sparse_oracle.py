"""Pins for the sparse (top-k) absorbed oracle ("One guard, 110x off the verify
step", section "The sparse model is different"): the full index list is the
dense attention, brute force on tiny inputs, order and padding do not matter,
the causal limit applies to listed positions, one position is its value.
CPU only."""

import math

import numpy as np
import pytest

from oracle import mla_oracle as O


def _case(rng, B, L, H, r, n, v, rope, lens):
    Tm = max(lens)
    return dict(q_nope=rng.standard_normal((B, L, H, n)), q_rope=rng.standard_normal((B, L, H, rope)),
                c_kv=rng.standard_normal((B, Tm, r)), k_rope=rng.standard_normal((B, Tm, rope)),
                W_UK=rng.standard_normal((H, n, r)) / math.sqrt(r),
                W_UV=rng.standard_normal((H, r, v)) / math.sqrt(r), cache_lens=lens)


def _brute_sparse(c, topk):
    """One score at a time over the listed, visible positions."""
    q_nope, q_rope, c_kv, k_rope = c["q_nope"], c["q_rope"], c["c_kv"], c["k_rope"]
    W_UK, W_UV = c["W_UK"], c["W_UV"]
    B, L, H, n = q_nope.shape
    s = 1.0 / math.sqrt(n + q_rope.shape[-1])
    out = np.zeros((B, L, H, W_UV.shape[-1]))
    for b in range(B):
        T = c["cache_lens"][b]
        for l in range(L):
            ts = [int(t) for t in topk[b][l] if 0 <= t <= T - L + l]
            for h in range(H):
                if not ts:
                    continue
                k = [W_UK[h] @ c_kv[b, t] for t in ts]
                sc = [s * (q_nope[b, l, h] @ k[i] + q_rope[b, l, h] @ k_rope[b, t])
                      for i, t in enumerate(ts)]
                m = max(sc)
                w = [math.exp(x - m) for x in sc]
                z = sum(w)
                for i, t in enumerate(ts):
                    out[b, l, h] += (w[i] / z) * (c_kv[b, t] @ W_UV[h])
    return out


def test_full_index_list_is_dense_attention():
    rng = np.random.default_rng(1)
    c = _case(rng, 2, 3, 2, 16, 8, 4, 4, [9, 20])
    topk = np.full((2, 3, 20), -1)
    for b, T in enumerate(c["cache_lens"]):
        topk[b, :, :T] = np.arange(T)
    np.testing.assert_allclose(O.sparse_absorbed(**c, topk=topk), O.absorbed(**c), atol=1e-12)


def test_sparse_matches_brute_force():
    rng = np.random.default_rng(2)
    c = _case(rng, 2, 3, 2, 8, 4, 3, 2, [11, 7])
    topk = np.stack([np.stack([rng.permutation(11)[:5] for _ in range(3)]) for _ in range(2)])
    np.testing.assert_allclose(O.sparse_absorbed(**c, topk=topk), _brute_sparse(c, topk),
                               atol=1e-12)


def test_order_and_padding_do_not_matter():
    rng = np.random.default_rng(3)
    c = _case(rng, 1, 2, 3, 16, 8, 4, 4, [30])
    base = np.stack([rng.permutation(29)[:6] for _ in range(2)])[None]
    shuffled = base[:, :, ::-1]
    padded = np.concatenate([np.full((1, 2, 3), -1), base, np.full((1, 2, 2), -1)], axis=2)
    want = O.sparse_absorbed(**c, topk=base)
    np.testing.assert_allclose(O.sparse_absorbed(**c, topk=shuffled), want, atol=1e-12)
    np.testing.assert_allclose(O.sparse_absorbed(**c, topk=padded), want, atol=1e-12)


def test_causal_limit_applies_to_listed_positions():
    # row l sees t <= T - L + l: the last position is listed for every row,
    # but only the last row may use it
    rng = np.random.default_rng(4)
    T, L = 12, 3
    c = _case(rng, 1, L, 2, 16, 8, 4, 4, [T])
    topk = np.array([[[0, 5, T - 1]] * L])
    got = O.sparse_absorbed(**c, topk=topk)
    np.testing.assert_allclose(got[:, :2], O.sparse_absorbed(**c, topk=topk[:, :, :2])[:, :2],
                               atol=1e-12)
    assert np.max(np.abs(got[:, 2] - O.sparse_absorbed(**c, topk=topk[:, :, :2])[:, 2])) > 1e-6


def test_single_position_is_its_value_and_empty_list_is_zero():
    rng = np.random.default_rng(5)
    c = _case(rng, 1, 2, 3, 16, 8, 4, 4, [10])
    topk = np.array([[[4, -1], [-1, -1]]])
    got = O.sparse_absorbed(**c, topk=topk)
    np.testing.assert_allclose(got[0, 0], np.einsum('r,hrv->hv', c["c_kv"][0, 4], c["W_UV"]),
                               atol=1e-12)
    assert np.all(got[0, 1] == 0)


def test_planted_causal_off_by_one_is_caught(monkeypatch):
    # a limit of t <= T - L + l + 1 (one position too far) must fail a pin
    real = O.sparse_absorbed

    def loose(**kw):
        kw["cache_lens"] = [int(t) + 1 for t in kw["cache_lens"]]
        return real(**kw)

    monkeypatch.setattr(O, "sparse_absorbed", loose)
    with pytest.raises(AssertionError):
        test_causal_limit_applies_to_listed_positions()
