"""Indexer key pooling with an incremental tail, and the top-k selection it
feeds (test infrastructure only).

Source: "One guard, 110x off the verify step" (stuartrowlands.com,
mla-absorbed-threshold):
* section "The same bug, one layer over": the sparse model's indexer pools
  the cached keys into windows of four before scoring them; completed
  windows are cached and only the tail is recomputed, for any number S of
  new tokens in a step (the defect was gating that on S == 1).  The guards
  that keep the incremental path correct: the cache has a pool, there is no
  padding, the batch shape matches, and the cache is exactly as long as the
  pool remembers (which catches a speculative rejection that trimmed the
  cache).  A wide step must pool exactly as the same tokens fed one at a
  time: window indices, cache length and the chosen top-k identical.
* section "The sparse model is different": the indexer selects the top 2048
  cached positions and attention runs over those only.

Readings taken where the page leaves a step open:
* A window w covers positions 4w .. 4w+3.  Its pooled key is the mean of the
  keys it holds; the last window of a cache whose length is not a multiple
  of four holds fewer than four (the tail) and is recomputed every step.
  Windows before floor(pool_len / 4) are complete and never change, because
  tokens only append.
* The incremental step recomputes windows floor(pool_len / 4) ..
  ceil(T / 4) - 1; any failed guard recomputes every window.
* Scoring: one indexer query vector per new token; window w's score is the
  dot product of the query with the pooled key.  Row s of a step sits at
  position T - S + s and may select window w when 4w <= T - S + s.  It keeps
  the k highest scores (ties to the lower window), listed by ascending
  window, and the attention list is those windows' positions 4w + i that the
  row may see, -1 padded to 4k entries.
The page gives no arithmetic beyond "windows of four", so these are the
plainest readings; 512 windows of four make the page's budget of 2048
positions.

parity pinned: tests/test_indexer_pool.py checks pooling against an explicit
per-window loop, a wide step against the same tokens fed one at a time and
against a fresh pool, each guard by breaking it, and the selection against
brute-force ranking on tiny inputs with the causal window limit.
"""

from __future__ import annotations

import numpy as np

WINDOW = 4


def num_windows(T: int) -> int:
    """Windows a cache of T tokens fills (the last one possibly partial)."""
    return (int(T) + WINDOW - 1) // WINDOW


def pool_window(keys, w: int, T: int):
    """Mean of the keys in window w of a cache of length T (float64)."""
    lo, hi = WINDOW * w, min(WINDOW * w + WINDOW, int(T))
    return np.asarray(keys[lo:hi], dtype=np.float64).mean(axis=0)


def pool_all(keys, T: int):
    """Pooled keys of every window of keys[:T] ([num_windows(T), d] float64)."""
    keys = np.asarray(keys, dtype=np.float64)
    return np.stack([pool_window(keys, w, T) for w in range(num_windows(T))]) \
        if T > 0 else np.zeros((0, keys.shape[-1]))


def pool_step(state, keys, T: int, S: int, padded: bool = False, batch: int = 1):
    """One indexer step over a cache that now holds T tokens, S of them new.

    ``state`` is None (no pool yet) or a dict {"pooled": [W, d], "length": L,
    "batch": b}.  Returns (new state, incremental?).  The incremental path
    keeps the windows completed at the remembered length and recomputes from
    the first window that was still open; every guard must hold for it."""
    keys = np.asarray(keys, dtype=np.float64)
    ok = (state is not None and not padded and state["batch"] == batch
          and state["length"] == T - S)
    if ok:
        keep = state["length"] // WINDOW          # windows complete before the step
        pooled = [state["pooled"][w] for w in range(keep)]
        pooled += [pool_window(keys, w, T) for w in range(keep, num_windows(T))]
        pooled = np.stack(pooled) if pooled else np.zeros((0, keys.shape[-1]))
    else:
        pooled = pool_all(keys, T)
    return {"pooled": pooled, "length": int(T), "batch": batch}, ok


def select_topk(q, pooled, T: int, S: int, k: int):
    """For each of the S new tokens, the k best visible windows and the
    positions they hold.  Returns (windows [S, k] int, positions [S, 4k] int),
    both -1 padded, windows ascending."""
    q = np.asarray(q, dtype=np.float64)
    pooled = np.asarray(pooled, dtype=np.float64)
    wins = np.full((S, k), -1, dtype=np.int64)
    pos = np.full((S, WINDOW * k), -1, dtype=np.int64)
    for s in range(S):
        p = T - S + s                          # this row's position
        vis = p // WINDOW + 1                  # windows w with 4w <= p
        scores = pooled[:vis] @ q[s]
        order = sorted(range(vis), key=lambda w: (-scores[w], w))[:k]
        chosen = sorted(order)
        wins[s, :len(chosen)] = chosen
        flat = [WINDOW * w + i for w in chosen for i in range(WINDOW) if WINDOW * w + i <= p]
        pos[s, :len(flat)] = flat
    return wins, pos
