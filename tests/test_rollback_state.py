"""Speculative-rollback state maintenance ("Over 107tok/s Qwen3.8-Flash-Next on
M3 Ultra", Algorithms 1, 4 and 5): the oracle against one-row-at-a-time
loops, the page's worked read count and every ValidBlock condition (CPU);
the library's kernels against the oracle bit for bit (GPU)."""

import numpy as np
import pytest
import torch

from oracle import rollback_state as O
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    yield


# ---------------------------------------------------------------------------
# Concatenation and snapshot windows
# ---------------------------------------------------------------------------

def _row_loop(S, T, X, cache, s, n, H, Q, ss, ts, xs, windows):
    """What Algorithm 5 says each thread stores, one row at a time."""
    for q in range(Q):
        for h in range(H):
            v = [S[i * ss[0] + h * ss[1] + q * ss[2]] for i in range(s)]
            v += [T[i * ts[0] + h * ts[1] + q * ts[2]] for i in range(n)]
            for i in range(s + n):
                X[i * xs[0] + h * xs[1] + q * xs[2]] = v[i]
            for a, off, stride in windows:
                for i in range(s):
                    cache[off + q * stride + h * s + i] = v[a + i]
    return X, cache


def _case(rng, s, n, H, Q, layout="row"):
    if layout == "row":           # [Q][H][i]
        ss, ts, xs = (1, s, H * s), (1, n, H * n), (1, s + n, H * (s + n))
    elif layout == "channels":    # channel-fastest new activations [Q][i][H]
        ss, ts, xs = (1, s, H * s), (H, 1, H * n), (1, s + n, H * (s + n))
    else:                         # channel-fastest state too: one thread per row
        ss, ts, xs = (H, 1, H * s), (H, 1, H * n), (1, s + n, H * (s + n))
    S = rng.integers(0, 2**32, size=H * Q * s, dtype=np.uint64).astype(np.uint32)
    T = rng.integers(0, 2**32, size=H * Q * n, dtype=np.uint64).astype(np.uint32)
    return S, T, ss, ts, xs


@pytest.mark.parametrize("layout", ["row", "channels"])
def test_separate_path_equals_row_loop(layout):
    rng = np.random.default_rng(1)
    s, n, H, Q = 3, 5, 7, 4
    S, T, ss, ts, xs = _case(rng, s, n, H, Q, layout)
    windows = [(0, 0, 3 * H * s), (2, H * s, 3 * H * s), (5, 2 * H * s, 3 * H * s)]
    cache_words = 3 * H * s * Q
    X1, c1 = O.concat_separate(S, T, np.zeros(H * Q * (s + n), np.uint32),
                               np.zeros(cache_words, np.uint32), s, n, H, Q, ss, ts, xs, windows)
    X2, c2 = _row_loop(S, T, np.zeros(H * Q * (s + n), np.uint32),
                       np.zeros(cache_words, np.uint32), s, n, H, Q, ss, ts, xs, windows)
    assert np.array_equal(X1, X2) and np.array_equal(c1, c2)


def test_worked_read_count():
    # "For an eight-element row and three snapshots of three elements each,
    # this reduces logical source reads from 17 to eight"
    assert O.logical_reads(3, 5, 3, fused=False) == 17
    assert O.logical_reads(3, 5, 3, fused=True) == 8


def test_fusion_checks():
    H, Q, s, n = 4, 2, 3, 5
    good = [(0, 0, 24), (1, 12, 24)]
    assert O.fusion_allowed(s, n, H, Q, good, 48, [])
    assert not O.fusion_allowed(s, n, H, Q, good[:1], 48, [])                 # k < 2
    assert not O.fusion_allowed(s, n, H, Q, [(0, 0, 24), (1, 6, 24)], 48, [])  # overlap
    assert not O.fusion_allowed(s, n, H, Q, [(0, 0, 24), (6, 12, 24)], 48, [])  # past the row
    assert not O.fusion_allowed(s, n, H, Q, good, 40, [])                      # past the cache
    assert not O.fusion_allowed(s, n, H, Q, good, 48, [(30, 31)])              # aliases a source
    assert not O.fusion_allowed(9, 5, H, Q, good, 48, [])                      # s > 8


# ---------------------------------------------------------------------------
# Rollback-valid prefix
# ---------------------------------------------------------------------------

def _chain(n_blocks, r):
    """Blocks of ratio r over cells 0..n_blocks*r-1 at their own positions."""
    cell_pos = np.arange(n_blocks * r, dtype=np.int32)
    cell_seq = np.ones(n_blocks * r, dtype=np.uint64)
    blocks = [dict(stream=0, start=b * r, src=list(range(b * r, b * r + r)), key=b * r,
                   pos=[b * r] * 4) for b in range(n_blocks)]
    return blocks, cell_pos, cell_seq


BREAKS = {
    "short source list": lambda b, cp, cs: b.update(src=b["src"][:-1]),
    "stream 1": lambda b, cp, cs: b.update(stream=1),
    "negative start": lambda b, cp, cs: b.update(start=-1),
    "key not a source": lambda b, cp, cs: b.update(key=10**6),
    "position component": lambda b, cp, cs: b["pos"].__setitem__(2, b["start"] + 1),
    "cell out of bounds": lambda b, cp, cs: b["src"].__setitem__(1, len(cp) + 3),
    "dead cell": lambda b, cp, cs: cp.__setitem__(b["src"][0], -1),
    "shared cell": lambda b, cp, cs: cs.__setitem__(b["src"][2], 3),
    "other sequence": lambda b, cp, cs: cs.__setitem__(b["src"][2], 2),
    "wrong position": lambda b, cp, cs: cp.__setitem__(b["src"][3], b["start"] + 7),
}


@pytest.mark.parametrize("what", sorted(BREAKS))
def test_each_valid_block_condition_stops_the_prefix(what):
    blocks, cp, cs = _chain(10, 4)
    assert O.retained_prefix(blocks, 4, 40, -1, cp, cs) == 10
    BREAKS[what](blocks[6], cp, cs)
    assert O.retained_prefix(blocks, 4, 40, -1, cp, cs) == 6


def test_prefix_stops_before_the_removed_suffix():
    # removal from p0 keeps the blocks ending at or before p0 (start + r <= p0):
    # the block [20, 24) survives a removal from 24, not one from 23
    blocks, cp, cs = _chain(10, 4)
    assert O.retained_prefix(blocks, 4, 24, -1, cp, cs) == 6
    assert O.retained_prefix(blocks, 4, 23, -1, cp, cs) == 5
    for g in [dict(streams=2), dict(seq=1)]:
        assert O.retained_prefix(blocks, 4, 40, -1, cp, cs, **g) == 0
    assert O.retained_prefix(blocks, 4, -1, -1, cp, cs) == 0
    assert O.retained_prefix(blocks, 4, 40, 50, cp, cs) == 0      # bounded removal


def test_retained_blocks_satisfy_the_invariant():
    # "Every retained block is complete, exclusively owned, and strictly before
    # the removed suffix" -- on random damage
    rng = np.random.default_rng(7)
    for _ in range(200):
        blocks, cp, cs = _chain(12, 4)
        for _ in range(int(rng.integers(0, 3))):
            BREAKS[sorted(BREAKS)[int(rng.integers(len(BREAKS)))]](
                blocks[int(rng.integers(12))], cp, cs)
        p0 = int(rng.integers(0, 60))
        k = O.retained_prefix(blocks, 4, p0, -1, cp, cs)
        for b in blocks[:k]:
            assert len(b["src"]) == 4 and b["start"] + 4 <= p0
            assert all(cs[c] == 1 and cp[c] == b["start"] + i for i, c in enumerate(b["src"]))


def test_planted_strict_suffix_bound_is_caught(monkeypatch):
    real = O.valid_block
    monkeypatch.setattr(O, "valid_block", lambda b, r, p0, cp, cs: real(b, r, p0 - 1, cp, cs))
    with pytest.raises(AssertionError):
        test_prefix_stops_before_the_removed_suffix()


# ---------------------------------------------------------------------------
# GPU: the library against the oracle, bit for bit
# ---------------------------------------------------------------------------

def _gpu_concat(rng, s, n, H, Q, windows, cache_words, layout="row"):
    S, T, ss, ts, xs = _case(rng, s, n, H, Q, layout)
    want_X, want_c = O.concat_separate(S, T, np.zeros(H * Q * (s + n), np.uint32),
                                       np.zeros(cache_words, np.uint32), s, n, H, Q, ss, ts,
                                       xs, windows)
    i32 = lambda a: torch.from_numpy(a.view(np.int32)).cuda()
    dS, dT = i32(S), i32(T)
    dX = torch.zeros(H * Q * (s + n), dtype=torch.int32, device="cuda")
    dc = torch.zeros(cache_words, dtype=torch.int32, device="cuda")
    fused = B.mla_concat_snapshots(dS, ss, dT, ts, dX, xs, s, n, H, Q, dc, windows)
    torch.cuda.synchronize()
    got_X = dX.cpu().numpy().view(np.uint32)
    got_c = dc.cpu().numpy().view(np.uint32)
    assert np.array_equal(got_X, want_X) and np.array_equal(got_c, want_c)
    return fused


@pytest.mark.gpu
@pytest.mark.parametrize("s,n,k,layout", [(3, 5, 3, "row"), (8, 8, 8, "row"), (1, 1, 2, "row"),
                                          (3, 6, 4, "channels"), (3, 5, 3, "planes"),
                                          (2, 7, 5, "planes")])
def test_gpu_fused_group_is_bit_exact(s, n, k, layout):
    rng = np.random.default_rng(s * 100 + n * 10 + k)
    H, Q = 300, 5
    block = k * H * s
    windows = [(int(rng.integers(0, n + 1)), j * H * s, block) for j in range(k)]
    assert _gpu_concat(rng, s, n, H, Q, windows, block * Q, layout)


@pytest.mark.gpu
@pytest.mark.parametrize("layout", ["row", "channels"])
@pytest.mark.parametrize("H", [3, 257, 515])
def test_gpu_padded_strides_and_ragged_runs_are_bit_exact(layout, H):
    # sequence strides padded to multiples of four words, so every run starts
    # on a 16-byte boundary and takes the 16-byte copies, while the channel
    # count leaves the last CTA's runs a few words past a multiple of four
    rng = np.random.default_rng(H + len(layout))
    s, n, k, Q = 3, 5, 3, 3
    pad = lambda x: (x + 7) // 4 * 4
    ss = (1, s, pad(H * s))
    ts = (1, n, pad(H * n)) if layout == "row" else (pad(H), 1, pad(H) * n + 4)
    xs = (1, s + n, pad(H * (s + n)))
    S = rng.integers(0, 2**32, size=ss[2] * Q, dtype=np.uint64).astype(np.uint32)
    T = rng.integers(0, 2**32, size=ts[2] * Q, dtype=np.uint64).astype(np.uint32)
    row = pad(H * s)
    block = k * row
    windows = [(int(rng.integers(0, n + 1)), j * row, block) for j in range(k)]
    want_X, want_c = O.concat_separate(S, T, np.zeros(xs[2] * Q, np.uint32),
                                       np.zeros(block * Q, np.uint32), s, n, H, Q, ss, ts, xs,
                                       windows)
    i32 = lambda a: torch.from_numpy(a.view(np.int32)).cuda()
    dX = torch.zeros(xs[2] * Q, dtype=torch.int32, device="cuda")
    dc = torch.zeros(block * Q, dtype=torch.int32, device="cuda")
    assert B.mla_concat_snapshots(i32(S), ss, i32(T), ts, dX, xs, s, n, H, Q, dc, windows)
    torch.cuda.synchronize()
    assert np.array_equal(dX.cpu().numpy().view(np.uint32), want_X)
    assert np.array_equal(dc.cpu().numpy().view(np.uint32), want_c)


@pytest.mark.gpu
def test_gpu_unsafe_group_takes_the_ordinary_path():
    rng = np.random.default_rng(3)
    s, n, H, Q = 3, 5, 64, 3
    # two windows writing the same words: the later one wins, as separate copies do
    windows = [(0, 0, H * s), (4, 0, H * s)]
    assert not _gpu_concat(rng, s, n, H, Q, windows, H * s * Q)
    assert not _gpu_concat(rng, s, n, H, Q, windows[:1], H * s * Q)       # one window


@pytest.mark.gpu
def test_gpu_window_outside_the_cache_is_rejected():
    d = torch.zeros(1024, dtype=torch.int32, device="cuda")
    with pytest.raises(B.MlaError):
        B.mla_concat_snapshots(d, (1, 3, 30), d, (1, 5, 50), d, (1, 8, 80), 3, 5, 10, 2,
                               torch.zeros(40, dtype=torch.int32, device="cuda"),
                               [(0, 0, 30), (1, 30, 30)])


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(6))
def test_gpu_rollback_prefix_matches_oracle(seed):
    rng = np.random.default_rng(100 + seed)
    r = 4
    n_blocks = int(rng.integers(1, 5000))
    blocks, cp, cs = _chain(n_blocks, r)
    for _ in range(int(rng.integers(0, 4))):
        BREAKS[sorted(BREAKS)[int(rng.integers(len(BREAKS)))]](
            blocks[int(rng.integers(n_blocks))], cp, cs)
    p0 = int(rng.integers(0, n_blocks * r + 8))
    want = O.retained_prefix(blocks, r, p0, -1, cp, cs)
    rows = np.full((n_blocks, 8 + r), -7, dtype=np.int32)
    for i, b in enumerate(blocks):
        rows[i, :8] = [b["stream"], b["start"], len(b["src"]), b["key"], *b["pos"]]
        rows[i, 8:8 + len(b["src"])] = b["src"][:r]
    got = B.mla_rollback_valid_prefix(torch.from_numpy(rows).cuda(), r,
                                      torch.from_numpy(cp).cuda(),
                                      torch.from_numpy(cs.view(np.int64)).cuda(), p0)
    assert int(got.item()) == want
    assert int(B.mla_rollback_valid_prefix(torch.from_numpy(rows).cuda(), r,
                                           torch.from_numpy(cp).cuda(),
                                           torch.from_numpy(cs.view(np.int64)).cuda(), p0,
                                           seq=1).item()) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(12))
def test_gpu_random_groups_are_bit_exact(i):
    # seeded random row widths, window counts and starts, channel and sequence
    # counts, all three layouts; one group in four gives two windows the same
    # destination, which must take the ordinary path with the same result
    rng = np.random.default_rng(300 + i)
    s = int(rng.integers(1, 9))
    n = int(rng.integers(1, 17 - s))
    k = int(rng.integers(1, 9))
    H = int(rng.integers(1, 700))
    Q = int(rng.integers(1, 7))
    layout = str(rng.choice(["row", "channels", "planes"]))
    block = k * H * s
    windows = [(int(rng.integers(0, n + 1)), j * H * s, block) for j in range(k)]
    unsafe = k >= 2 and rng.random() < 0.25
    if unsafe:
        windows[1] = (windows[1][0], windows[0][1], block)
    fused = _gpu_concat(rng, s, n, H, Q, windows, block * Q, layout)
    assert fused == (k >= 2 and not unsafe)
