"""Float64 CPU oracle for MLA verify attention (test infrastructure only).

This module is the plain, slow, obviously-correct statement of what the GPU
library computes.  It exists so that tests, the smoke check and the CPU
baseline leg of the benchmark have something independent to compare against.
Nothing in the product path imports it, and it imports nothing from the
product: it needs only numpy (and, optionally, the caller's arrays).

Sources (web pages, cited by title and section):

* "One guard, 110x off the verify step. Speculative decoding on MLA models in
  MLX" (stuartrowlands.com, mla-absorbed-threshold):
  - section "The defect": the two mathematically equivalent ways to use a
    compressed latent cache -- absorbed (fold the up-projection into the
    query, attend against the latent) and materialised (expand the cache to
    full K and V, attend normally).
  - section "The threshold is not a constant": the per-head cost model and
    the long-cache limit r(n+v)/(2r-n-v), with the table of thresholds
    170 / 398 / 512.
  - section "The change": the helper that floors the limit, returns 1 when
    the denominator is not positive, and never returns less than 1; the
    guard "L <= max_absorbed".
* "fix: Speed up multi-token decode by computing the absorbed MLA threshold"
  (mlx-lm pull request 1817):
  - opening section: the finite-cache crossover L < r*d/(r*d/T + 2r - d),
    d = n + v, and the cold-cache reversal at T == L.
  - section "Where the paths cross": 379 at cache 8192 for 512/192/256.
  - reviewer comment: use exact integer arithmetic for the crossover.

Readings taken where the pages leave a step open (each also listed in the
design notes of the repository):

* T is the cache length *including* the L new rows; row l of a verify block
  sits at position T - L + l and sees positions 0 .. T - L + l (causal among
  the verify rows).
* The guard is "L <= floor(x)" (ties go to the absorbed branch), as in the
  helper's code, which is what makes the printed 512 for 512/256/256 hold.
* With a non-positive denominator the helper's answer (1) is used for the
  finite-cache form as well.
* A batch of sequences makes one decision from the summed cost model:
  L <= floor(r*d*sum(T) / (B*r*d + (2r-d)*sum(T))), which is the pages'
  formula when B == 1.
* The softmax scale is a parameter (1/sqrt(n + rope) by default); RoPE is
  already applied to q_rope and k_rope.

parity pinned: every function here is checked in tests/test_oracle.py against
something other than itself -- the printed thresholds, brute force on tiny
inputs, torch's scaled_dot_product_attention (its default scale is the
query width's inverse square root, which pins default_scale), the absorbed ==
materialised identity, closed-form special cases, and for gather_paged a
round trip through an independently written page scatter plus paged ==
contiguous attention under a random page permutation.
"""

from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

MODE_AUTO = 0
MODE_ABSORBED = 1
MODE_MATERIALISED = 2

BRANCH_ABSORBED = 1
BRANCH_MATERIALISED = 2


# ---------------------------------------------------------------------------
# Crossover threshold
# ---------------------------------------------------------------------------

def max_absorbed_queries(r: int, n: int, v: int, cache_len: int | None = None) -> int:
    """Largest number of query rows for which the absorbed branch is cheaper.

    Cost model per head ("The threshold is not a constant"): the absorbed
    branch does 2*L*T*r work on attention plus L*r*d on the fold; the
    materialised branch does T*r*d to expand plus L*T*d to attend
    (d = n + v).  Setting them equal gives

        L = r*d*T / (r*d + (2r - d)*T)            (finite cache, pull request text)
        L = r*d / (2r - d)                        (T -> infinity, the helper)

    ``cache_len`` None (or <= 0) asks for the limit.  Exact rational
    arithmetic is used (reviewer comment on the pull request), then floored;
    a non-positive denominator gives 1, and the result is never below 1
    ("The change").
    """
    r, n, v = int(r), int(n), int(v)
    d = n + v
    if cache_len is None or int(cache_len) <= 0:
        denom = 2 * r - d
        if denom <= 0:
            return 1
        x = Fraction(r * d, denom)
    else:
        t = int(cache_len)
        if 2 * r - d <= 0:
            return 1
        denom = r * d + (2 * r - d) * t
        x = Fraction(r * d * t, denom)
    return max(1, math.floor(x))


def max_absorbed_queries_batch(r: int, n: int, v: int, cache_lens) -> int:
    """One decision for a batch: the summed cost model (B == 1 gives the pages' formula).

    Summing the per-sequence costs of "The threshold is not a constant" over
    the batch: absorbed L*(2r*sum(T) + B*r*d), materialised
    sum(T)*r*d + L*sum(T)*d; equal at L = r*d*S / (B*r*d + (2r-d)*S).
    """
    lens = [int(t) for t in cache_lens]
    if len(lens) == 1:
        return max_absorbed_queries(r, n, v, lens[0])
    r, n, v = int(r), int(n), int(v)
    d = n + v
    if 2 * r - d <= 0:
        return 1
    s = sum(lens)
    b = len(lens)
    x = Fraction(r * d * s, b * r * d + (2 * r - d) * s)
    return max(1, math.floor(x))


def select_branch(r: int, n: int, v: int, L: int, cache_lens, mode: int = MODE_AUTO) -> int:
    """Branch the guard "L <= max_absorbed" picks ("The change"); forced modes override."""
    if mode == MODE_ABSORBED:
        return BRANCH_ABSORBED
    if mode == MODE_MATERIALISED:
        return BRANCH_MATERIALISED
    thr = max_absorbed_queries_batch(r, n, v, cache_lens)
    return BRANCH_ABSORBED if int(L) <= thr else BRANCH_MATERIALISED


# ---------------------------------------------------------------------------
# Attention, both branches
# ---------------------------------------------------------------------------

def default_scale(n: int, rope: int) -> float:
    """Softmax scale 1/sqrt(n + rope): the query/key width the scores are taken over."""
    return 1.0 / math.sqrt(n + rope)


def _causal_mask(T: int, L: int) -> np.ndarray:
    """[L, T] boolean: row l (at position T-L+l) may see key positions t <= T-L+l."""
    t = np.arange(T)[None, :]
    last = (T - L + np.arange(L))[:, None]
    return t <= last


def _softmax_rows(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis (masked entries hold -inf)."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def absorbed(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, scale=None,
             heads=None, rows=None, head_chunk=16):
    """Absorbed branch ("The defect", first bullet).

    Shapes: q_nope [B,L,H,n], q_rope [B,L,H,rope], c_kv [B,Tmax,r],
    k_rope [B,Tmax,rope], W_UK [H,n,r], W_UV [H,r,v], cache_lens [B].
    Returns out [B,len(rows),len(heads),v] in float64 (``heads`` / ``rows``
    select a subset of heads / verify rows; every output is independent).

    Steps: q_lat = q_nope . W_UK (fold, n -> r); scores = scale*(q_lat . c_kv^T
    + q_rope . k_rope^T) with the causal verify mask; softmax; o_lat =
    P . c_kv (accumulated in the latent space); out = o_lat . W_UV (r -> v).
    """
    q_nope, q_rope = _as64(q_nope), _as64(q_rope)
    W_UK, W_UV = _as64(W_UK), _as64(W_UV)
    B, L, H, n = q_nope.shape
    rope = q_rope.shape[-1]
    v = W_UV.shape[-1]
    if scale is None:
        scale = default_scale(n, rope)
    heads = list(range(H)) if heads is None else list(heads)
    rows = list(range(L)) if rows is None else list(rows)
    out = np.zeros((B, len(rows), len(heads), v), dtype=np.float64)
    for b in range(B):
        T = int(cache_lens[b])
        ckv = _as64(c_kv[b, :T])     # [T, r]   (converted one sequence at a time)
        kr = _as64(k_rope[b, :T])    # [T, rope]
        mask = _causal_mask(T, L)[rows]   # [rows, T]
        for c0 in range(0, len(heads), head_chunk):
            hs = heads[c0:c0 + head_chunk]
            qn = q_nope[b][rows][:, hs]               # [rows, h, n]
            qr = q_rope[b][rows][:, hs]               # [rows, h, rope]
            q_lat = np.einsum('lhn,hnr->hlr', qn, W_UK[hs])          # fold
            s = (q_lat @ ckv.T + np.einsum('lhp,tp->hlt', qr, kr)) * scale
            s = np.where(mask[None], s, -np.inf)
            p = _softmax_rows(s)                      # [h, L, T]
            o_lat = p @ ckv                           # [h, L, r]
            o = np.einsum('hlr,hrv->lhv', o_lat, W_UV[hs])           # unembed
            out[b, :, c0:c0 + len(hs)] = o
    return out


def materialised(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, scale=None,
                 heads=None, rows=None, head_chunk=8):
    """Materialised branch ("The defect", second bullet).

    Expand the cached latent to full per-head keys K_nope = c_kv . W_UK^T and
    values V = c_kv . W_UV, then ordinary causal attention with the query
    [q_nope || q_rope] against [K_nope || k_rope] (the RoPE key is shared by
    all heads).  Same shapes and return as :func:`absorbed`.
    """
    q_nope, q_rope = _as64(q_nope), _as64(q_rope)
    W_UK, W_UV = _as64(W_UK), _as64(W_UV)
    B, L, H, n = q_nope.shape
    rope = q_rope.shape[-1]
    v = W_UV.shape[-1]
    if scale is None:
        scale = default_scale(n, rope)
    heads = list(range(H)) if heads is None else list(heads)
    rows = list(range(L)) if rows is None else list(rows)
    out = np.zeros((B, len(rows), len(heads), v), dtype=np.float64)
    for b in range(B):
        T = int(cache_lens[b])
        ckv = _as64(c_kv[b, :T])
        kr = _as64(k_rope[b, :T])
        mask = _causal_mask(T, L)[rows]
        for c0 in range(0, len(heads), head_chunk):
            hs = heads[c0:c0 + head_chunk]
            k_nope = np.einsum('tr,hnr->htn', ckv, W_UK[hs])       # expand keys
            val = np.einsum('tr,hrv->htv', ckv, W_UV[hs])          # expand values
            qn = np.transpose(q_nope[b][rows][:, hs], (1, 0, 2))   # [h, rows, n]
            qr = q_rope[b][rows][:, hs]
            s = (qn @ np.transpose(k_nope, (0, 2, 1))
                 + np.einsum('lhp,tp->hlt', qr, kr)) * scale
            s = np.where(mask[None], s, -np.inf)
            p = _softmax_rows(s)
            o = p @ val                                            # [h, rows, v]
            out[b, :, c0:c0 + len(hs)] = np.transpose(o, (1, 0, 2))
    return out


def brute_force(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, scale=None):
    """Attention written out one score at a time with Python loops (tiny inputs only).

    For each sequence b, verify row l and head h: the key of cached position t
    is k_t = W_UK[h] c_kv[t] (n values) next to k_rope[t]; the value is
    u_t = c_kv[t] W_UV[h].  The score is scale*(q_nope.k_t + q_rope.k_rope[t])
    over the visible positions t <= T-L+l, and the output is the softmax-
    weighted sum of the u_t.  No matrix routine, no branch logic.
    """
    q_nope, q_rope, c_kv, k_rope = map(_as64, (q_nope, q_rope, c_kv, k_rope))
    W_UK, W_UV = _as64(W_UK), _as64(W_UV)
    B, L, H, n = q_nope.shape
    rope = q_rope.shape[-1]
    r = c_kv.shape[-1]
    v = W_UV.shape[-1]
    if scale is None:
        scale = default_scale(n, rope)
    out = np.zeros((B, L, H, v), dtype=np.float64)
    for b in range(B):
        T = int(cache_lens[b])
        for l in range(L):
            last = T - L + l
            for h in range(H):
                scores = []
                for t in range(last + 1):
                    acc = 0.0
                    for i in range(n):
                        k_ti = 0.0
                        for j in range(r):
                            k_ti += W_UK[h, i, j] * c_kv[b, t, j]
                        acc += q_nope[b, l, h, i] * k_ti
                    for p in range(rope):
                        acc += q_rope[b, l, h, p] * k_rope[b, t, p]
                    scores.append(acc * scale)
                mx = max(scores)
                w = [math.exp(s - mx) for s in scores]
                z = sum(w)
                for t in range(last + 1):
                    a = w[t] / z
                    for k in range(v):
                        u = 0.0
                        for j in range(r):
                            u += c_kv[b, t, j] * W_UV[h, j, k]
                        out[b, l, h, k] += a * u
    return out


def gather_paged(pages, page_table, cache_lens, page_size):
    """Contiguous per-sequence rows from a paged cache.

    pages [num_pages, page_size, w]; page_table [B, max_pages] int; sequence b's
    position t lives in page page_table[b, t // page_size], row t % page_size.
    Returns [B, max(cache_lens), w] with rows past each length left at zero.
    """
    pages = np.asarray(pages)
    B = len(cache_lens)
    Tmax = int(max(cache_lens))
    out = np.zeros((B, Tmax, pages.shape[-1]), dtype=pages.dtype)
    for b in range(B):
        T = int(cache_lens[b])
        t = np.arange(T)
        out[b, :T] = pages[np.asarray(page_table)[b, t // page_size], t % page_size]
    return out


def sparse_absorbed(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, topk, scale=None,
                    heads=None, rows=None):
    """Absorbed attention over a selected set of cached positions.

    "One guard, 110x off the verify step", section "The sparse model is
    different": an indexer selects the top 2048 cached positions and attention
    runs over those only.  ``topk`` [B, L, k] lists, for verify row l of
    sequence b, the positions its attention reads; an entry is used when
    0 <= t <= T_b - L + l (the causal verify limit), so -1 pads a short list.
    Readings: every head of a verify row shares its list (the indexer picks
    positions, the heads share the latent); a row whose list holds no usable
    position returns zeros.  Otherwise the steps are those of ``absorbed``,
    with the scores taken over the listed positions only.
    """
    q_nope, q_rope = _as64(q_nope), _as64(q_rope)
    W_UK, W_UV = _as64(W_UK), _as64(W_UV)
    topk = np.asarray(topk)
    B, L, H, n = q_nope.shape
    rope = q_rope.shape[-1]
    v = W_UV.shape[-1]
    if scale is None:
        scale = default_scale(n, rope)
    heads = list(range(H)) if heads is None else list(heads)
    rows = list(range(L)) if rows is None else list(rows)
    out = np.zeros((B, len(rows), len(heads), v), dtype=np.float64)
    for b in range(B):
        T = int(cache_lens[b])
        for ri, l in enumerate(rows):
            idx = [int(t) for t in topk[b, l] if 0 <= int(t) <= T - L + l]
            if not idx:
                continue
            ckv = _as64(c_kv[b, idx])          # [k', r]
            kr = _as64(k_rope[b, idx])         # [k', rope]
            qn = q_nope[b, l, heads]           # [h, n]
            qr = q_rope[b, l, heads]           # [h, rope]
            q_lat = np.einsum('hn,hnr->hr', qn, W_UK[heads])
            s_ = (q_lat @ ckv.T + qr @ kr.T) * scale
            p_ = _softmax_rows(s_)
            o_lat = p_ @ ckv
            out[b, ri] = np.einsum('hr,hrv->hv', o_lat, W_UV[heads])
    return out