"""Seeded synthetic inputs for MLA verify attention.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic, so both the float64 oracle and the CUDA library can be
fed from it.  The pages measure on real checkpoints (GLM-4.7-Flash,
Moonlight-16B, Kimi-Linear) that are not available here; these draws stand in
for them with the same geometry:

* activations q_nope, q_rope, c_kv, k_rope ~ N(0, 1);
* weights W_UK, W_UV ~ N(0, 1/512) (standard deviation 1/sqrt(512));
* all draws are float32 from a ``torch.Generator`` seeded per case (on the
  CPU, or on the GPU for the benchmark's large shapes), then rounded to the
  case's dtype (bf16 rounds to nearest even).

Layouts (row-major): q_nope [B,L,H,n], q_rope [B,L,H,rope],
c_kv [B,Tmax,r], k_rope [B,Tmax,rope], W_UK [H,n,r], W_UV [H,r,v].
A paged cache stores c_kv as [num_pages, page_size, r] and k_rope as
[num_pages, page_size, rope] with an int32 page table [B, max_pages].
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Geometry:
    H: int
    r: int = 512
    n: int = 128
    v: int = 128
    rope: int = 64

    @property
    def d(self) -> int:
        return self.n + self.v


DSV3 = Geometry(H=128, r=512, n=128, v=128, rope=64)      # 512/128/128, threshold 170
GLM47 = Geometry(H=32, r=512, n=192, v=256, rope=64)      # 512/192/256, threshold 398
GLM53 = Geometry(H=64, r=512, n=256, v=256, rope=64)      # 512/256/256, threshold 512
TINY = Geometry(H=4, r=512, n=128, v=128, rope=64)


@dataclasses.dataclass
class Case:
    """One verify call's inputs (CPU tensors), plus the metadata to rebuild it."""
    geom: Geometry
    L: int
    cache_lens: list
    dtype: torch.dtype
    q_nope: torch.Tensor
    q_rope: torch.Tensor
    c_kv: torch.Tensor          # contiguous [B,Tmax,r] or paged [P,page,r]
    k_rope: torch.Tensor        # contiguous [B,Tmax,rope] or paged [P,page,rope]
    W_UK: torch.Tensor
    W_UV: torch.Tensor
    page_table: Optional[torch.Tensor] = None   # int32 [B, max_pages] when paged
    page_size: int = 0

    @property
    def B(self) -> int:
        return len(self.cache_lens)

    @property
    def paged(self) -> bool:
        return self.page_table is not None


def _normal(gen, shape, std, dtype):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32, device=gen.device)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def dominant_position(T: int, L: int) -> int:
    """Where ``make_case(dominant=...)`` plants its key: position T - L + 1, the
    first one that verify row 0 must not see (T // 2 when L == 1)."""
    return T - L + 1 if L > 1 else T // 2


def make_case(geom: Geometry, L: int, cache_lens, dtype=torch.bfloat16, seed: int = 0,
              page_size: int = 0, tmax: Optional[int] = None, q_std: float = 1.0,
              dominant: float = 0.0, device="cpu") -> Case:
    """Draw one case.  ``page_size`` > 0 gives a paged cache with a random page table.

    Draw order is fixed (q_nope, q_rope, cache, k_rope, W_UK, W_UV, page
    permutation) so a seed names one input set for a given shape.
    Contiguous caches are [B, Tmax, *] with Tmax = max(cache_lens) unless
    ``tmax`` is given; paged caches hold sum(ceil(T_b/page)) pages, shuffled,
    and the tail rows of each sequence's last page are filled with random
    values too (they must be ignored by the attention).

    Sharper score distributions for edge cases: ``q_std`` scales both query
    parts (q_std = 12 gives scores with a standard deviation of about 12
    nats at the configured geometries instead of about 1); ``dominant`` = D > 0
    sets the first RoPE component of every query to D and that of the key at
    ``dominant_position(T_b, L)`` to D, so that key wins by about D^2/sqrt(n+rope)
    nats (contiguous caches only).

    ``device`` draws on that device with its own seeded generator (a CUDA
    generator gives other values than the CPU one for the same seed; the
    benchmark draws its large inputs this way, the tests on the CPU).
    """
    cache_lens = [int(t) for t in cache_lens]
    B = len(cache_lens)
    g = torch.Generator(device=device).manual_seed(int(seed))
    wstd = 1.0 / (512 ** 0.5)
    q_nope = _normal(g, (B, L, geom.H, geom.n), q_std, dtype)
    q_rope = _normal(g, (B, L, geom.H, geom.rope), q_std, dtype)
    page_table = None
    if page_size > 0:
        npages = [(t + page_size - 1) // page_size for t in cache_lens]
        total = sum(npages)
        c_kv = _normal(g, (total, page_size, geom.r), 1.0, dtype)
        k_rope = _normal(g, (total, page_size, geom.rope), 1.0, dtype)
    else:
        tm = max(cache_lens) if tmax is None else int(tmax)
        c_kv = _normal(g, (B, tm, geom.r), 1.0, dtype)
        k_rope = _normal(g, (B, tm, geom.rope), 1.0, dtype)
    W_UK = _normal(g, (geom.H, geom.n, geom.r), wstd, dtype)
    W_UV = _normal(g, (geom.H, geom.r, geom.v), wstd, dtype)
    if page_size > 0:
        perm = torch.randperm(total, generator=g, device=g.device).to(torch.int32)
        maxp = max(npages)
        page_table = torch.zeros((B, maxp), dtype=torch.int32, device=g.device)
        k = 0
        for b in range(B):
            page_table[b, :npages[b]] = perm[k:k + npages[b]]
            k += npages[b]
    if dominant:
        if page_size > 0:
            raise ValueError("dominant keys are planted in contiguous caches only")
        q_rope[..., 0] = dominant
        for b, T in enumerate(cache_lens):
            k_rope[b, dominant_position(T, L), 0] = dominant
    return Case(geom, L, cache_lens, dtype, q_nope, q_rope, c_kv, k_rope, W_UK, W_UV,
                page_table, page_size)


def uniform_cache_lens(B: int, lo: int, hi: int, seed: int) -> list:
    """Seeded integer draw T_b ~ U{lo..hi} (batched serving mix)."""
    g = torch.Generator().manual_seed(int(seed) + 7919)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


# Workload recipes: the five configurations the measurements are quoted on.
WORKLOADS = {
    # tiny fp32 layer: H=4, 512/128/128, one sequence, T=512, L=4
    "tiny_fp32": dict(geom=TINY, dtype=torch.float32, seed=0,
                      shapes=[(4, [512])]),
    # DeepSeek-V3-like geometry, B=1, T in {512,2048,8192}, L in {1,2,4,8,16}
    "dsv3": dict(geom=DSV3, dtype=torch.bfloat16, seed=1,
                 shapes=[(L, [T]) for T in (512, 2048, 8192) for L in (1, 2, 4, 8, 16)]),
    # GLM-4.7-Flash-like geometry, T=8192, branch-crossover sweep
    "glm47_sweep": dict(geom=GLM47, dtype=torch.bfloat16, seed=2,
                        shapes=[(L, [8192]) for L in
                                (1, 16, 64, 128, 256, 379, 398, 512, 1024, 2048)]),
    # batched serving verify: 32 sequences, T_b ~ U{1024..32768}, L=8, paged (64)
    "batched_paged": dict(geom=DSV3, dtype=torch.bfloat16, seed=3, page_size=64,
                          shapes=[(8, "uniform:32:1024:32768")]),
    # long-context verify, 512/256/256, H=64, B=4, T=131072; cold prefill T=L=2048
    "long_context": dict(geom=GLM53, dtype=torch.bfloat16, seed=4,
                         shapes=[(L, [131072] * 4) for L in (1, 5, 8, 16)]
                         + [(2048, [2048] * 4)]),
}


def workload_shapes(name: str):
    """Expand a recipe into (L, cache_lens) pairs."""
    w = WORKLOADS[name]
    out = []
    for L, lens in w["shapes"]:
        if isinstance(lens, str):
            _, B, lo, hi = lens.split(":")
            lens = uniform_cache_lens(int(B), int(lo), int(hi), w["seed"])
        out.append((L, list(lens)))
    return out


def make_topk(cache_lens, L: int, k: int, seed: int, pad: int = 0, past_limit: int = 0,
              device="cpu") -> torch.Tensor:
    """Seeded synthetic index lists for the sparse (top-k) call: int32
    [B, L, k].  Row l of sequence b lists k distinct positions drawn uniformly
    from [0, T_b) (all of them, in random order, padded with -1 when k > T_b),
    a stand-in for an indexer's selection; then the last ``pad`` entries of
    every list become -1 and ``past_limit`` entries (when there are that many
    positions past the row's causal limit T_b - L + l) are swapped for such
    positions, which the attention must skip."""
    B = len(cache_lens)
    g = torch.Generator().manual_seed(int(seed) + 104729)
    out = torch.full((B, L, k), -1, dtype=torch.int32)
    for b, T in enumerate(cache_lens):
        for l in range(L):
            perm = torch.randperm(int(T), generator=g)[:k].to(torch.int32)
            out[b, l, :perm.numel()] = perm
            last = int(T) - L + l
            beyond = torch.arange(last + 1, int(T), dtype=torch.int32)
            m = min(int(past_limit), beyond.numel(), k)
            if m:
                out[b, l, :m] = beyond[:m]
            if pad:
                out[b, l, k - min(pad, k):] = -1
    return out.to(device)
