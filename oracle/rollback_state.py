"""Speculative-rollback state maintenance (test infrastructure only).

Source: "Over 107tok/s Qwen3.8-Flash-Next on M3 Ultra" (blog.salty.li):
* section "A later extension: load snapshot history once", Algorithm 4
  (recognise a safe snapshot group) and Algorithm 5 (materialise the
  concatenation and every snapshot window from one load per row);
* section "Keep the pooled keys; score them again", the predicate
  ValidBlock and Algorithm 1 (retain a rollback-valid prefix).

Concatenation and snapshot windows.  State S (s words per channel/sequence
row), new activations T (n words per row), H channels, Q sequences.  Element
i of row (h, q) of a buffer with strides (di, dh, dq) sits at word
i*di + h*dh + q*dq.  The concatenation is X[i, h, q] = S[i, h, q] for i < s
and T[i - s, h, q] for s <= i < s + n.  A window descriptor (a, offset,
stride) copies X[a .. a+s-1, h, q] to cache words offset + q*stride + h*s + i
(the page's d[h s + i]).  The ordinary path is the page's "separate passes":
write X, then one copy per window that reads X again.  Words are copied as
bit patterns (uint32), never as floats.

Readings taken where the page leaves a step open:
* Window starts satisfy 0 <= a and a + s <= s + n (a window lies inside the
  concatenated row).
* Algorithm 4's checks are: 1 <= s, n <= 8, s + n <= 16, 2 <= k <= 8
  windows, every destination word inside the cache, destinations of
  different windows disjoint, and no destination inside S, T or X (given as
  word ranges).  When they fail, the ordinary path runs instead.

Rollback-valid prefix.  Cells carry a logical position (negative: empty)
and the set of sequences that own them (a bit mask).  A pooled block of
ratio r carries its stream, start, source cells, key destination cell and
four stored positional components.  ValidBlock(b, r, p0) holds when the
block has exactly r source cells, stream 0, start >= 0, start + r <= p0, its
key cell is one of its source cells, all four positional components equal
the start, and source cell i is inside the cell array, live, owned by
sequence 0 alone, and at logical position start + i.  Algorithm 1 keeps the
longest prefix of blocks that pass, stopping at the first that does not;
when a global guard fails (streams != 1, sequence != 0, p0 < 0, or a bounded
removal p1 >= 0) nothing is kept.

parity pinned: tests/test_rollback_state.py checks the ordinary path
against a one-row-at-a-time loop of what Algorithm 5 says each thread
stores, the page's worked count (an eight-word row and three
three-word snapshots: 17 logical reads separately, 8 fused), every
ValidBlock condition broken one at a time, and the stated invariant that
every retained block is complete, exclusively owned and before the suffix.
"""

from __future__ import annotations

import numpy as np


# ---------------------------------------------------------------------------
# Concatenation and snapshot windows
# ---------------------------------------------------------------------------

def _index(shape_i, H, Q, strides):
    di, dh, dq = strides
    i = np.arange(shape_i)[:, None, None]
    h = np.arange(H)[None, :, None]
    q = np.arange(Q)[None, None, :]
    return i * di + h * dh + q * dq     # [i, h, q] word offsets


def concat_separate(S, T, X, cache, s, n, H, Q, s_strides, t_strides, x_strides, windows):
    """The ordinary path: write X = S || T, then one copy per window reading X.

    S, T, X, cache are flat uint32 arrays (X and cache are written in place);
    windows is a list of (a, offset, stride).  Returns (X, cache)."""
    X[_index(s, H, Q, x_strides)] = S[_index(s, H, Q, s_strides)]
    xi = _index(s + n, H, Q, x_strides)
    X[xi[s:]] = T[_index(n, H, Q, t_strides)]
    for a, offset, stride in windows:
        src = X[xi[a:a + s]]                                  # [s, H, Q]
        i = np.arange(s)[:, None, None]
        h = np.arange(H)[None, :, None]
        q = np.arange(Q)[None, None, :]
        cache[offset + q * stride + h * s + i] = src
    return X, cache


def logical_reads(s, n, k, fused):
    """Source words read per row: s + n once when fused, s + n + k*s when each
    snapshot rereads the concatenation (Algorithm 5's cost argument)."""
    return s + n if fused else s + n + k * s


def _ranges_overlap(ranges):
    """True when any two half-open word ranges [lo, hi) overlap."""
    rs = sorted(r for r in ranges if r[1] > r[0])
    return any(b[0] < a[1] for a, b in zip(rs, rs[1:]))


def fusion_allowed(s, n, H, Q, windows, cache_words, other_ranges):
    """Algorithm 4's safety checks (see the module doc); other_ranges are the
    word ranges of S, T and X in the same address space as the cache."""
    if not (1 <= s <= 8 and 1 <= n <= 8 and s + n <= 16):
        return False
    if not (2 <= len(windows) <= 8):
        return False
    dest = []
    for a, offset, stride in windows:
        if a < 0 or a + s > s + n or offset < 0 or stride < 0:
            return False
        if offset + (Q - 1) * stride + H * s > cache_words:
            return False
        dest.append([(offset + q * stride, offset + q * stride + H * s) for q in range(Q)])
    for j in range(len(dest)):
        if _ranges_overlap(dest[j]):       # one window's rows must not overlap either
            return False
    flat = [r for d in dest for r in d]
    if _ranges_overlap(flat):
        return False
    for lo, hi in other_ranges:            # no destination inside S, T or X
        if any(a < hi and lo < b for a, b in flat):
            return False
    return True


# ---------------------------------------------------------------------------
# Rollback-valid prefix
# ---------------------------------------------------------------------------

def valid_block(block, r, p0, cell_pos, cell_seq):
    """ValidBlock(b, r, p0, M) for one block (a dict with stream, start,
    src (list of cell ids), key, pos (four ints))."""
    src = list(block["src"])
    if len(src) != r or block["stream"] != 0 or block["start"] < 0:
        return False
    if block["start"] + r > p0:
        return False
    if block["key"] not in src:
        return False
    if any(c != block["start"] for c in block["pos"]):
        return False
    for i, c in enumerate(src):
        if not (0 <= c < len(cell_pos)):
            return False
        if cell_pos[c] < 0:                      # not live
            return False
        if int(cell_seq[c]) != 1:                # owned by sequence 0 alone
            return False
        if cell_pos[c] != block["start"] + i:
            return False
    return True


def retained_prefix(blocks, r, p0, p1, cell_pos, cell_seq, seq=0, streams=1):
    """Algorithm 1 for one pooling ratio: how many leading blocks stay valid."""
    if streams != 1 or seq != 0 or p0 < 0 or p1 >= 0:
        return 0
    k = 0
    for b in blocks:
        if not valid_block(b, r, p0, cell_pos, cell_seq):
            break
        k += 1
    return k
