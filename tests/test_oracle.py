"""Pins for the float64 oracle: printed values, brute force, a library routine,
the branch identity and closed forms.  CPU only."""

import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import mla_oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))


def _golden_thresholds():
    rows = []
    with open(os.path.join(HERE, "golden", "thresholds.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            r, n, v, t, want, src = line.split(None, 5)
            rows.append((int(r), int(n), int(v), None if t == "inf" else int(t), int(want), src))
    return rows


# ---------------------------------------------------------------------------
# Threshold
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("r,n,v,t,want,src", _golden_thresholds())
def test_threshold_printed_values(r, n, v, t, want, src):
    assert oracle.max_absorbed_queries(r, n, v, t) == want, src


def test_threshold_cold_cache_reverses():
    # pull request opening section: with T == L the materialised branch always wins
    for (r, n, v) in [(512, 128, 128), (512, 192, 256), (512, 256, 256), (256, 64, 64)]:
        for L in (2, 3, 16, 512, 2048, 4096):
            assert oracle.select_branch(r, n, v, L, [L]) == oracle.BRANCH_MATERIALISED
    # L == 1 is always absorbed (the helper never returns less than 1)
    assert oracle.select_branch(512, 128, 128, 1, [1]) == oracle.BRANCH_ABSORBED


def test_threshold_cold_prefill_case():
    # the long-context cold prefill case T = L = 2048 on 512/256/256 must materialise
    assert oracle.select_branch(512, 256, 256, 2048, [2048] * 4) == oracle.BRANCH_MATERIALISED


def test_threshold_degenerate_denominator():
    # "The change": a non-positive denominator gives 1
    assert oracle.max_absorbed_queries(64, 64, 64) == 1          # 2r - d == 0
    assert oracle.max_absorbed_queries(64, 100, 100) == 1        # 2r - d < 0
    assert oracle.max_absorbed_queries(64, 64, 64, 4096) == 1


def test_threshold_finite_tends_to_limit():
    # the finite-cache form grows with T and never exceeds the long-cache limit
    for (r, n, v) in [(512, 128, 128), (512, 192, 256), (512, 256, 256)]:
        lim = oracle.max_absorbed_queries(r, n, v)
        prev = 0
        for t in [1, 2, 8, 64, 512, 4096, 8192, 65536, 1 << 20, 1 << 30]:
            x = oracle.max_absorbed_queries(r, n, v, t)
            assert prev <= x <= lim
            prev = x
        assert oracle.max_absorbed_queries(r, n, v, 1 << 40) >= lim - 1


def test_threshold_exact_at_integer_quotient():
    # 512/256/256 in the limit is exactly 512.0: ties go to absorbed (printed 512).
    assert oracle.max_absorbed_queries(512, 256, 256) == 512
    # any finite cache stays strictly below the limit here
    assert oracle.max_absorbed_queries(512, 256, 256, 1 << 40) == 511
    # DeepSeek-V3 geometry at T = 512: r*d*T / (r*d + (2r-d)*T) = 67108864/524288 = 128 exactly
    assert oracle.max_absorbed_queries(512, 128, 128, 512) == 128
    assert oracle.select_branch(512, 128, 128, 128, [512]) == oracle.BRANCH_ABSORBED
    assert oracle.select_branch(512, 128, 128, 129, [512]) == oracle.BRANCH_MATERIALISED


def test_threshold_cost_model_brute_force():
    # The threshold is the largest L at which absorbed cost <= materialised cost, with the
    # per-head costs of "The threshold is not a constant" counted term by term.
    def absorbed_cost(L, T, r, n, v):
        return 2 * L * T * r + L * r * (n + v)

    def materialised_cost(L, T, r, n, v):
        return T * r * (n + v) + L * T * (n + v)

    for (r, n, v) in [(512, 128, 128), (512, 192, 256), (512, 256, 256), (96, 40, 24)]:
        for T in (1, 7, 100, 512, 2048, 8192):
            best = 0
            for L in range(1, 4096):
                if absorbed_cost(L, T, r, n, v) <= materialised_cost(L, T, r, n, v):
                    best = L
            assert oracle.max_absorbed_queries(r, n, v, T) == max(1, best), (r, n, v, T)


def test_threshold_batch_summed_cost():
    # one decision per batch from the summed costs; equal lengths and B == 1 reduce to the
    # single-sequence value
    for T in (512, 2048, 8192):
        assert oracle.max_absorbed_queries_batch(512, 128, 128, [T] * 7) == \
            oracle.max_absorbed_queries(512, 128, 128, T)
    lens = [1000, 5000, 20000, 333]
    r, n, v = 512, 192, 256
    d = n + v
    best = 0
    for L in range(1, 2000):
        a = sum(2 * L * T * r + L * r * d for T in lens)
        m = sum(T * r * d + L * T * d for T in lens)
        if a <= m:
            best = L
    assert oracle.max_absorbed_queries_batch(r, n, v, lens) == best


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _rand_case(rng, B, L, H, r, n, v, rope, lens, wstd=None):
    Tmax = max(lens)
    wstd = wstd if wstd is not None else 1.0 / math.sqrt(r)
    return dict(
        q_nope=rng.standard_normal((B, L, H, n)),
        q_rope=rng.standard_normal((B, L, H, rope)),
        c_kv=rng.standard_normal((B, Tmax, r)),
        k_rope=rng.standard_normal((B, Tmax, rope)),
        W_UK=rng.standard_normal((H, n, r)) * wstd,
        W_UV=rng.standard_normal((H, r, v)) * wstd,
        cache_lens=lens,
    )


def test_brute_force_matches_both_branches_tiny():
    rng = np.random.default_rng(11)
    c = _rand_case(rng, B=2, L=3, H=2, r=8, n=4, v=3, rope=2, lens=[5, 7])
    bf = O.brute_force(**c)
    a = O.absorbed(**c)
    m = O.materialised(**c)
    np.testing.assert_allclose(a, bf, rtol=0, atol=1e-12)
    np.testing.assert_allclose(m, bf, rtol=0, atol=1e-12)


def test_brute_force_scale_parameter():
    rng = np.random.default_rng(12)
    c = _rand_case(rng, B=1, L=2, H=2, r=6, n=3, v=4, rope=2, lens=[4])
    for s in (0.37, 2.0):
        np.testing.assert_allclose(O.absorbed(**c, scale=s), O.brute_force(**c, scale=s),
                                   atol=1e-12)


def _sdpa_reference(c, scale=None):
    """Same attention through torch's scaled_dot_product_attention (float64, CPU).

    ``scale`` None leaves the scale to the library, whose default is the
    inverse square root of the query width, here n + rope: an independent
    statement of the oracle's default_scale."""
    q_nope, q_rope = c["q_nope"], c["q_rope"]
    B, L, H, n = q_nope.shape
    out = np.zeros((B, L, H, c["W_UV"].shape[-1]))
    for b in range(B):
        T = c["cache_lens"][b]
        ckv = torch.from_numpy(c["c_kv"][b, :T])
        kr = torch.from_numpy(c["k_rope"][b, :T])
        for h in range(H):
            k = torch.cat([ckv @ torch.from_numpy(c["W_UK"][h]).T, kr], dim=1)   # [T, n+rope]
            val = ckv @ torch.from_numpy(c["W_UV"][h])                             # [T, v]
            q = torch.cat([torch.from_numpy(q_nope[b, :, h]),
                           torch.from_numpy(q_rope[b, :, h])], dim=1)              # [L, n+rope]
            allow = torch.zeros((L, T), dtype=torch.bool)
            for l in range(L):
                allow[l, :T - L + l + 1] = True
            o = torch.nn.functional.scaled_dot_product_attention(
                q[None, None], k[None, None], val[None, None], attn_mask=allow[None, None],
                scale=scale)
            out[b, :, h] = o[0, 0].numpy()
    return out


@pytest.mark.parametrize("geom", [(512, 128, 128), (512, 192, 256), (512, 256, 256)])
def test_branches_match_library_attention(geom):
    r, n, v = geom
    rng = np.random.default_rng(r + n + v)
    c = _rand_case(rng, B=2, L=5, H=3, r=r, n=n, v=v, rope=64, lens=[37, 80])
    ref = _sdpa_reference(c)      # the library's own default scale
    np.testing.assert_allclose(O.absorbed(**c), ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(O.materialised(**c), ref, atol=1e-12, rtol=0)


def test_absorbed_equals_materialised_configured_geometry():
    # "The defect": the two ways to use the cache are mathematically equivalent
    rng = np.random.default_rng(5)
    c = _rand_case(rng, B=3, L=16, H=8, r=512, n=192, v=256, rope=64, lens=[16, 300, 1025])
    a = O.absorbed(**c)
    m = O.materialised(**c)
    assert np.max(np.abs(a - m)) < 1e-12
    assert np.max(np.abs(a)) > 1e-3


def test_head_subset_matches_full():
    rng = np.random.default_rng(6)
    c = _rand_case(rng, B=2, L=4, H=10, r=64, n=16, v=8, rope=4, lens=[20, 33])
    full = O.absorbed(**c)
    sub = O.absorbed(**c, heads=[9, 2, 5])
    np.testing.assert_array_equal(sub, full[:, :, [9, 2, 5]])
    subm = O.materialised(**c, heads=[1, 7])
    np.testing.assert_allclose(subm, full[:, :, [1, 7]], atol=1e-12)
    rows = O.absorbed(**c, heads=[3, 4], rows=[3, 0])
    np.testing.assert_allclose(rows, full[:, [3, 0]][:, :, [3, 4]], atol=1e-14)
    rowsm = O.materialised(**c, heads=[8], rows=[2])
    np.testing.assert_allclose(rowsm, full[:, [2]][:, :, [8]], atol=1e-12)


def test_closed_form_single_position():
    # T = L = 1: the only visible key is position 0, so out = c_kv[0] . W_UV
    rng = np.random.default_rng(7)
    c = _rand_case(rng, B=2, L=1, H=4, r=32, n=8, v=6, rope=4, lens=[1, 1])
    want = np.einsum('br,hrv->bhv', c["c_kv"][:, 0], c["W_UV"])[:, None]
    for fn in (O.absorbed, O.materialised):
        np.testing.assert_allclose(fn(**c), want, atol=1e-12)


def test_closed_form_constant_latent():
    # every cached latent row equal to c: any softmax weights give c . W_UV
    rng = np.random.default_rng(8)
    c = _rand_case(rng, B=1, L=3, H=3, r=32, n=8, v=5, rope=4, lens=[9])
    row = rng.standard_normal(32)
    c["c_kv"][:] = row
    want = np.broadcast_to(np.einsum('r,hrv->hv', row, c["W_UV"]), (1, 3, 3, 5))
    for fn in (O.absorbed, O.materialised):
        np.testing.assert_allclose(fn(**c), want, atol=1e-12)


def test_closed_form_zero_query_uniform_prefix_mean():
    # q = 0: all visible scores are 0, so row l averages positions 0..T-L+l
    rng = np.random.default_rng(9)
    c = _rand_case(rng, B=2, L=4, H=2, r=16, n=8, v=3, rope=4, lens=[6, 11])
    c["q_nope"][:] = 0
    c["q_rope"][:] = 0
    out = O.absorbed(**c)
    for b, T in enumerate(c["cache_lens"]):
        for l in range(4):
            mean = c["c_kv"][b, :T - 4 + l + 1].mean(axis=0)
            want = np.einsum('r,hrv->hv', mean, c["W_UV"])
            np.testing.assert_allclose(out[b, l], want, atol=1e-12)
    np.testing.assert_allclose(O.materialised(**c), out, atol=1e-12)


def test_closed_form_zero_latent():
    rng = np.random.default_rng(10)
    c = _rand_case(rng, B=1, L=2, H=2, r=16, n=4, v=3, rope=4, lens=[5])
    c["c_kv"][:] = 0
    for fn in (O.absorbed, O.materialised):
        assert np.all(fn(**c) == 0)


def test_causal_mask_boundary_with_dominant_key():
    # one key made overwhelmingly attractive through the RoPE part, at position T-L+1:
    # rows l >= 1 see it (output = its value), row 0 must not (mask offset T-L+l).
    rng = np.random.default_rng(13)
    T, L = 10, 4
    c = _rand_case(rng, B=1, L=L, H=2, r=16, n=4, v=3, rope=4, lens=[T])
    c["q_nope"] *= 1e-3
    c["k_rope"][:] = 0
    star = T - L + 1
    c["k_rope"][0, star, 0] = 40.0
    c["q_rope"][:] = 0
    c["q_rope"][..., 0] = 40.0
    val = np.einsum('r,hrv->hv', c["c_kv"][0, star], c["W_UV"])
    for fn in (O.absorbed, O.materialised):
        out = fn(**c)
        for l in range(1, L):
            np.testing.assert_allclose(out[0, l], val, atol=1e-9)
        assert np.max(np.abs(out[0, 0] - val)) > 1e-3


def _scatter_to_pages(contig, lens, page, perm):
    """The inverse of a page walk, written independently of gather_paged:
    sequence b's logical page j (rows j*page .. j*page+page-1 of its
    contiguous cache) is copied whole into physical page perm[k], k counting
    pages in sequence order.  Returns (pages, page table)."""
    npg = [-(-T // page) for T in lens]
    pages = np.full((sum(npg), page, contig.shape[-1]), np.nan)
    table = np.full((len(lens), max(npg)), -1, dtype=np.int64)
    k = 0
    for b, T in enumerate(lens):
        for j in range(npg[b]):
            dst = int(perm[k])
            k += 1
            table[b, j] = dst
            rows = contig[b, j * page:min((j + 1) * page, T)]
            pages[dst, :rows.shape[0]] = rows
    return pages, table


def test_gather_paged_round_trip():
    # scatter a contiguous cache into shuffled pages, gather it back: exact
    rng = np.random.default_rng(14)
    for page, lens in ((4, [5, 9, 1]), (64, [64, 65, 200, 3]), (16, [16, 1, 47])):
        contig = rng.standard_normal((len(lens), max(lens), 3))
        perm = rng.permutation(sum(-(-T // page) for T in lens))
        pages, table = _scatter_to_pages(contig, lens, page, perm)
        got = O.gather_paged(pages, table, lens, page)
        for b, T in enumerate(lens):
            assert np.array_equal(got[b, :T], contig[b, :T])


def test_paged_attention_equals_contiguous():
    # attention over a paged cache (gathered) equals attention over the
    # contiguous cache, for a random page permutation
    rng = np.random.default_rng(17)
    page = 8
    c = _rand_case(rng, B=3, L=3, H=2, r=16, n=8, v=4, rope=4, lens=[9, 24, 3])
    perm = rng.permutation(sum(-(-T // page) for T in c["cache_lens"]))
    pc, table = _scatter_to_pages(c["c_kv"], c["cache_lens"], page, perm)
    pk, _ = _scatter_to_pages(c["k_rope"], c["cache_lens"], page, perm)
    paged = dict(c, c_kv=O.gather_paged(pc, table, c["cache_lens"], page),
                 k_rope=O.gather_paged(pk, table, c["cache_lens"], page))
    np.testing.assert_array_equal(O.absorbed(**paged), O.absorbed(**c))
    np.testing.assert_allclose(O.brute_force(**paged), O.absorbed(**c), atol=1e-12)


def test_default_scale_stated_value():
    # the tiny fp32 workload states its softmax scale as 1/sqrt(192) for
    # n = 128, rope = 64 (the pages themselves leave the scale open)
    assert O.default_scale(128, 64) == 1.0 / math.sqrt(192)
    assert abs(O.default_scale(128, 64) - 0.07216878364870323) < 1e-17


# ---------------------------------------------------------------------------
# The pins bite: a planted mistake in the oracle must fail at least one of them
# ---------------------------------------------------------------------------

def test_planted_mask_offset_is_caught(monkeypatch):
    rng = np.random.default_rng(15)
    c = _rand_case(rng, B=1, L=3, H=2, r=8, n=4, v=3, rope=2, lens=[6])
    good = O.brute_force(**c)

    def shifted(T, L):
        t = np.arange(T)[None, :]
        return t <= (T - L + np.arange(L))[:, None] - 1 + (np.arange(L)[:, None] == 0)

    monkeypatch.setattr(O, "_causal_mask", shifted)
    assert np.max(np.abs(O.absorbed(**c) - good)) > 1e-3


def test_planted_scale_is_caught(monkeypatch):
    # 1/sqrt(n) instead of 1/sqrt(n + rope): caught by the stated literal and by
    # the library attention's default scale
    rng = np.random.default_rng(16)
    c = _rand_case(rng, B=1, L=2, H=2, r=512, n=128, v=128, rope=64, lens=[20])
    ref = _sdpa_reference(c)
    monkeypatch.setattr(O, "default_scale", lambda n, rope: 1.0 / math.sqrt(n))
    assert np.max(np.abs(O.absorbed(**c) - ref)) > 1e-4
    with pytest.raises(AssertionError):
        test_default_scale_stated_value()


def test_planted_threshold_strictness_is_caught(monkeypatch):
    # a strict "<" guard would make the printed 512 for 512/256/256 come out 511
    real = O.max_absorbed_queries

    def strict(r, n, v, cache_len=None):
        x = real(r, n, v, cache_len)
        d = n + v
        exact = (cache_len is None and (r * d) % (2 * r - d) == 0)
        return x - 1 if exact else x

    monkeypatch.setattr(O, "max_absorbed_queries", strict)
    rows = [g for g in _golden_thresholds() if g[:3] == (512, 256, 256)]
    assert any(O.max_absorbed_queries(r, n, v, t) != want for r, n, v, t, want, _ in rows)


def test_planted_page_walk_off_by_one_is_caught(monkeypatch):
    real = O.gather_paged

    def off_by_one(pages, page_table, cache_lens, page_size):
        pages = np.asarray(pages)
        out = np.zeros((len(cache_lens), int(max(cache_lens)), pages.shape[-1]))
        for b, T in enumerate(cache_lens):
            t = np.arange(int(T))
            out[b, :T] = pages[np.asarray(page_table)[b, (t + 1) // page_size], t % page_size]
        return out

    monkeypatch.setattr(O, "gather_paged", off_by_one)
    with pytest.raises(AssertionError):
        test_gather_paged_round_trip()
    monkeypatch.setattr(O, "gather_paged", real)
    test_gather_paged_round_trip()
