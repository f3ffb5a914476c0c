"""GPU checks of the indexer pooling and top-k window selection against the
float64 oracle ("One guard, 110x off the verify step", section "The same
bug, one layer over"): pooled keys within fp32 rounding of the oracle's
means; a wide step bit for bit equal to the same tokens fed one at a time and
to a fresh pool, at aligned and misaligned cache lengths; each guard forcing
a full recompute; the incremental step reusing completed windows; the chosen
windows a valid top-k (exactly the oracle's wherever the k-th score is not a
near tie); and the chosen positions feeding the sparse verify call."""

import numpy as np
import pytest
import torch

import oracle
from oracle import indexer_pool as P
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import DSV3, make_case
from parity_util import compare, device_tensors, oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    B.lib()
    yield


def _keys(B_, T, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B_, T, d, generator=g).to(dtype)


def _pool(keys, T, S, pooled, state, **kw):
    inc = B.mla_indexer_pool_update(keys, T, S, pooled, state, **kw)
    torch.cuda.synchronize()
    return inc


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_pool_matches_oracle(dtype):
    keys = _keys(2, 1003, 128, dtype, 1)
    kd = keys.cuda()
    pooled = torch.full((2, 260, 128), float("nan"), device="cuda")
    st = B.IndexerPoolState()
    assert not _pool(kd, 1003, 1003, pooled, st)
    assert (st.length, st.batch, st.dim) == (1003, 2, 128)
    for b in range(2):
        want = P.pool_all(keys[b].double().numpy(), 1003)
        got = pooled[b, :want.shape[0]].double().cpu().numpy()
        np.testing.assert_allclose(got, want, rtol=2e-7, atol=2e-7)
    assert torch.isnan(pooled[:, 251:]).all()   # windows past the cache untouched


@pytest.mark.parametrize("S", [2, 3, 4, 8])
@pytest.mark.parametrize("T0", [4096, 4097, 4098, 4099])
def test_wide_step_equals_one_at_a_time(S, T0):
    keys = _keys(1, T0 + S, 128, torch.bfloat16, S * 10 + T0).cuda()
    W = -(-(T0 + S) // 4)

    def start():
        pooled = torch.zeros((1, W + 4, 128), device="cuda")
        st = B.IndexerPoolState()
        _pool(keys, T0, T0, pooled, st)
        return pooled, st

    wide, sw = start()
    assert _pool(keys, T0 + S, S, wide, sw)
    one, so = start()
    for t in range(T0 + 1, T0 + S + 1):
        assert _pool(keys, t, 1, one, so)
    fresh = torch.zeros_like(wide)
    _pool(keys, T0 + S, T0 + S, fresh, B.IndexerPoolState())
    assert torch.equal(wide[:, :W], one[:, :W])
    assert torch.equal(wide[:, :W], fresh[:, :W])
    assert sw.length == so.length == T0 + S


def test_incremental_step_reuses_completed_windows():
    keys = _keys(1, 300, 64, torch.float32, 5).cuda()
    pooled = torch.zeros((1, 80, 64), device="cuda")
    st = B.IndexerPoolState()
    _pool(keys, 290, 290, pooled, st)
    before = pooled.clone()
    keys[:, :288] += 100.0        # windows 0..71 were complete at 290
    assert _pool(keys, 300, 10, pooled, st)
    assert torch.equal(pooled[:, :72], before[:, :72])
    fresh = torch.zeros_like(pooled)
    _pool(keys, 300, 300, fresh, B.IndexerPoolState())
    assert torch.equal(pooled[:, 72:75], fresh[:, 72:75])


@pytest.mark.parametrize("guard", ["trim", "padded", "batch", "fresh"])
def test_guards_force_a_full_recompute(guard):
    keys = _keys(2, 64, 64, torch.float32, 9).cuda()
    pooled = torch.zeros((2, 16, 64), device="cuda")
    st = B.IndexerPoolState()
    _pool(keys, 40, 40, pooled, st)
    kw, T, S = {}, 42, 2
    if guard == "trim":
        T = 39                    # a rejection trimmed 40 -> 37, then 2 new tokens
        keys[:, 37:39] = -keys[:, 37:39]
    elif guard == "padded":
        kw["padded"] = True
    elif guard == "batch":
        st.batch = 1
    else:
        st = B.IndexerPoolState()
    assert not _pool(keys, T, S, pooled, st, **kw)
    fresh = torch.zeros_like(pooled)
    _pool(keys, T, T, fresh, B.IndexerPoolState())
    W = -(-T // 4)
    assert torch.equal(pooled[:, :W], fresh[:, :W])


def _check_selection(q, pooled, T, S, k, wins, pos):
    """Valid top-k under float64 scores of the GPU's pooled keys; exactly the
    oracle's choice where the k-th score is not within rounding of the next."""
    q64 = q.double().cpu().numpy()
    pk = pooled.double().cpu().numpy()
    wins, pos = wins.cpu().numpy(), pos.cpu().numpy()
    for b in range(q64.shape[0]):
        W_ = -(-T // 4)
        ow, opos = P.select_topk(q64[b], pk[b, :W_], T, S, k)
        for s in range(S):
            p = T - S + s
            vis = p // 4 + 1
            got = [int(w) for w in wins[b, s] if w >= 0]
            assert len(got) == min(k, vis) and got == sorted(got) and all(w < vis for w in got)
            sc = pk[b, :vis] @ q64[b, s]
            tol = 1e-4 * max(1.0, float(np.abs(sc).max()))
            chosen = np.zeros(vis, bool)
            chosen[got] = True
            if (~chosen).any():
                assert sc[chosen].min() >= sc[~chosen].max() - tol
                ranked = np.sort(sc)[::-1]
                if ranked[len(got) - 1] - ranked[len(got)] > tol:
                    assert got == [int(w) for w in ow[s] if w >= 0]
            flat = [4 * w + i for w in got for i in range(4) if 4 * w + i <= p]
            assert list(pos[b, s, :len(flat)]) == flat and np.all(pos[b, s, len(flat):] == -1)
            if got == [int(w) for w in ow[s] if w >= 0]:
                assert np.array_equal(pos[b, s], opos[s])


@pytest.mark.parametrize("T,S,k", [(4099, 4, 64), (131072, 8, 512), (37, 3, 20), (9, 2, 512),
                                   (200003, 2, 1000)])
def test_select_is_a_valid_topk(T, S, k):
    keys = _keys(2, T, 128, torch.bfloat16, T + S).cuda()
    pooled = torch.zeros((2, -(-T // 4), 128), device="cuda")
    _pool(keys, T, T, pooled, B.IndexerPoolState())
    g = torch.Generator().manual_seed(7 * T)
    q = torch.randn(2, S, 128, generator=g).cuda()
    wins, pos = B.mla_indexer_select(q, pooled, T, k)
    torch.cuda.synchronize()
    _check_selection(q, pooled, T, S, k, wins, pos)


@pytest.mark.parametrize("T,S,k,dim", [(5003, 3, 200, 64), (9001, 20, 300, 96),
                                       (131075, 4, 512, 128), (200003, 2, 3000, 64),
                                       (1048803, 2, 700, 32)])
def test_select_with_many_ties_is_exactly_the_oracles(T, S, k, dim):
    # small-integer keys and queries: every score is an exact fp32 integer
    # whatever the summation order, so many windows tie at the k-th score and
    # the choice (ties to the lower window) is unique.  A row of windows is
    # spread over a cluster of CTAs up to 262120 windows; 1048803 tokens make
    # 262201, which one CTA per row selects over several output rounds, from
    # global memory.  dim 96 and 32 take the scoring kernel's generic form
    g = torch.Generator().manual_seed(T + k)
    W = -(-T // 4)
    pooled = torch.randint(-3, 4, (1, W, dim), generator=g).float()
    q = torch.randint(-2, 3, (1, S, dim), generator=g).float()
    wins, pos = B.mla_indexer_select(q.cuda(), pooled.cuda(), T, k)
    torch.cuda.synchronize()
    ow, opos = P.select_topk(q[0].double().numpy(), pooled[0].double().numpy(), T, S, k)
    assert np.array_equal(wins[0].cpu().numpy(), ow)
    assert np.array_equal(pos[0].cpu().numpy(), opos)


@pytest.mark.parametrize("T,S,dim", [(4099, 9, 128), (150, 17, 128), (4099, 9, 64)])
def test_pool_rows_past_the_cache_are_never_read_into_the_choice(T, S, dim):
    # a pool with room for more windows than the cache fills, the rest NaN:
    # the scoring reads whole tiles of rows (those past the last window are
    # scored and dropped), and the choice must equal the oracle's on the
    # filled rows exactly (small-integer data, exact scores)
    g = torch.Generator().manual_seed(T + S)
    W = -(-T // 4)
    filled = torch.randint(-3, 4, (2, W, dim), generator=g).float()
    pooled = torch.full((2, W + 100, dim), float("nan"))
    pooled[:, :W] = filled
    q = torch.randint(-2, 3, (2, S, dim), generator=g).float()
    wins, pos = B.mla_indexer_select(q.cuda(), pooled.cuda(), T, 300)
    torch.cuda.synchronize()
    for b in range(2):
        ow, opos = P.select_topk(q[b].double().numpy(), filled[b].double().numpy(), T, S, 300)
        assert np.array_equal(wins[b].cpu().numpy(), ow)
        assert np.array_equal(pos[b].cpu().numpy(), opos)


def test_selection_ties_go_to_the_lower_window():
    pooled = torch.ones((1, 10, 32), device="cuda")
    q = torch.ones((1, 1, 32), device="cuda")
    wins, pos = B.mla_indexer_select(q, pooled, 40, 3)
    torch.cuda.synchronize()
    assert wins.cpu().tolist() == [[[0, 1, 2]]]
    assert pos.cpu().tolist() == [[list(range(12))]]


def test_selected_positions_feed_the_sparse_verify():
    # pool -> select (512 windows = 2048 positions) -> sparse attention
    T, L = 8192, 2
    case = make_case(DSV3, L, [T], seed=61)
    keys = _keys(1, T, 128, torch.bfloat16, 61).cuda()
    pooled = torch.zeros((1, T // 4, 128), device="cuda")
    _pool(keys, T, T, pooled, B.IndexerPoolState())
    q = torch.randn(1, L, 128, generator=torch.Generator().manual_seed(62)).cuda()
    _, pos = B.mla_indexer_select(q, pooled, T, 512)
    d = device_tensors(case)
    out = B.mla_verify_attention_sparse(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"],
                                        d["W_UK"], d["W_UV"], case.cache_lens, pos,
                                        cache_lens_dev=d["lens_dev"])
    torch.cuda.synchronize()
    heads = [0, 5, 127]
    want = oracle.sparse_absorbed(**oracle_inputs(case), topk=pos.cpu().numpy(), heads=heads)
    compare(out[:, :, heads], want, torch.bfloat16, "indexer -> sparse verify")


def _select_draw(i):
    rng = np.random.default_rng(8000 + i)
    T = int(np.exp(rng.uniform(np.log(1), np.log(300000))))
    dim = int(rng.choice([32, 64, 96, 128, 128, 256]))
    S = int(rng.integers(1, min(32, 48 * 1024 // (4 * dim)) + 1))
    S = min(S, T)
    k = int(rng.integers(1, 4001))
    batch = int(rng.integers(1, 4))
    return T, S, k, dim, batch


@pytest.mark.parametrize("i", range(16))
def test_random_select_is_exactly_the_oracles(i):
    # seeded random shapes with small-integer keys and queries (every score an
    # exact fp32 integer, many ties): the chosen windows and positions equal
    # the oracle's bit for bit, through either form of the selection
    T, S, k, dim, batch = _select_draw(i)
    g = torch.Generator().manual_seed(8100 + i)
    W = -(-T // 4)
    pooled = torch.randint(-3, 4, (batch, W, dim), generator=g).float()
    q = torch.randint(-2, 3, (batch, S, dim), generator=g).float()
    wins, pos = B.mla_indexer_select(q.cuda(), pooled.cuda(), T, k)
    torch.cuda.synchronize()
    for b in range(batch):
        ow, opos = P.select_topk(q[b].double().numpy(), pooled[b].double().numpy(), T, S, k)
        assert np.array_equal(wins[b].cpu().numpy(), ow), (i, T, S, k, dim, b)
        assert np.array_equal(pos[b].cpu().numpy(), opos), (i, T, S, k, dim, b)
