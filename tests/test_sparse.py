"""GPU parity of the sparse (top-k) verify call against the float64 oracle.

"One guard, 110x off the verify step", section "The sparse model is
different": an indexer selects the top 2048 cached positions and attention
runs over those only.  mla_verify_attention_sparse takes one index list per
verify row; the oracle's sparse_absorbed is the dense absorbed attention
restricted to the listed positions that the row may see.  The tensor-core
kernel (H a multiple of 128) gathers the listed rows tile by tile; other
geometries and fp32 run the CUDA-core kernels.  Cases span several 64-entry
tiles and a ragged tail, padding, positions past a row's causal limit, paged
caches, empty lists, and the full-size DeepSeek-V3-like shape (k = 2048 at
T = 8192 and 32768, sampled heads).
"""

import numpy as np
import pytest
import torch

import oracle
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import DSV3, GLM53, TINY, Geometry, make_case, make_topk
from parity_util import compare, device_tensors, oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    B.lib()
    yield


def run_sparse(case, topk, **kw):
    d = device_tensors(case)
    out = B.mla_verify_attention_sparse(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"],
                                        d["W_UK"], d["W_UV"], case.cache_lens, topk.cuda(),
                                        page_table=d["page_table"],
                                        cache_lens_dev=d["lens_dev"], **kw)
    torch.cuda.synchronize()
    B.mla_device_status()
    return out


def want_sparse(case, topk, heads=None, rows=None):
    inp = oracle_inputs(case)
    return oracle.sparse_absorbed(**inp, topk=topk.numpy(), heads=heads, rows=rows)


def kernels_of(fn):
    B.mla_kernel_timing_read(reset=True)
    B.mla_kernel_timing_enable(True)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        B.mla_kernel_timing_enable(False)
    return out, set(B.mla_kernel_timing_read(reset=True))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_tiny_generic(dtype):
    case = make_case(TINY, 4, [512], dtype=dtype, seed=0)
    topk = make_topk([512], 4, 96, seed=0, pad=7, past_limit=2)
    got = run_sparse(case, topk)
    compare(got, want_sparse(case, topk), dtype, f"tiny sparse {dtype}")


@pytest.mark.parametrize("L,T,k,seed", [(1, 8192, 2048, 1), (4, 32768, 2048, 2)])
def test_dsv3_full_size(L, T, k, seed):
    # the tensor-core path at the sparse model's budget; every head of every
    # row is compared on a sample of heads
    case = make_case(DSV3, L, [T], seed=seed)
    topk = make_topk([T], L, k, seed=seed, past_limit=3 if L > 1 else 0)
    got, names = kernels_of(lambda: run_sparse(case, topk))
    assert "absorbed_attn_sparse_sm103" in names, names
    heads = [0, 1, 63, 64, 127]
    want = want_sparse(case, topk, heads=heads)
    compare(got[:, :, heads], want, torch.bfloat16, f"dsv3 sparse L={L} T={T}")


@pytest.mark.parametrize("L,lens,k,page", [
    (2, [3000, 700], 1000, 64),   # ragged last tile (1000 = 15 * 64 + 40), paged
    (3, [130, 5000], 70, 0),      # 64 + 6 entries, lists longer than a short cache
    (1, [9000], 5, 0),            # a single partial tile
])
def test_fast_ragged_and_paged(L, lens, k, page):
    case = make_case(Geometry(H=128), L, lens, seed=11 + k, page_size=page)
    topk = make_topk(lens, L, k, seed=k, pad=3, past_limit=1)
    got, names = kernels_of(lambda: run_sparse(case, topk))
    assert "absorbed_attn_sparse_sm103" in names, names
    compare(got, want_sparse(case, topk), torch.bfloat16, f"sparse L={L} lens={lens} k={k}")


def test_empty_and_single_position_lists():
    # row 0: nothing usable (zeros); row 1: one position (its value row);
    # row 2: a normal list
    lens = [4000]
    case = make_case(Geometry(H=128), 3, lens, seed=21)
    topk = make_topk(lens, 3, 200, seed=21)
    topk[0, 0, :] = -1
    topk[0, 1, :] = -1
    topk[0, 1, 77] = 1234
    got = run_sparse(case, topk)
    want = want_sparse(case, topk)
    assert np.all(want[0, 0] == 0.0)
    assert torch.all(got[0, 0] == 0)
    compare(got, want, torch.bfloat16, "empty / single-position lists")


def test_generic_fallback_geometry():
    # 64 heads: a 128-row tile would hold two verify rows' lists, so the
    # CUDA-core kernels run
    case = make_case(GLM53, 2, [4096], seed=31)
    topk = make_topk([4096], 2, 512, seed=31, pad=5, past_limit=1)
    got, names = kernels_of(lambda: run_sparse(case, topk))
    assert "generic_absorbed_attention" in names and "absorbed_attn_sparse_sm103" not in names
    compare(got, want_sparse(case, topk), torch.bfloat16, "sparse generic 512/256/256")


def test_full_list_matches_dense_call():
    # every position listed, in order: the dense call's attention
    T, L = 1500, 2
    case = make_case(Geometry(H=128), L, [T], seed=41)
    topk = torch.arange(T, dtype=torch.int32).repeat(1, L, 1)
    got = run_sparse(case, topk)
    d = device_tensors(case)
    dense, _ = B.mla_verify_attention(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"],
                                      d["W_UK"], d["W_UV"], case.cache_lens, mode="absorbed",
                                      cache_lens_dev=d["lens_dev"])
    torch.cuda.synchronize()
    want = want_sparse(case, topk)
    compare(got, want, torch.bfloat16, "full list vs oracle")
    compare(dense, want, torch.bfloat16, "dense vs oracle")


def test_repeat_call_is_deterministic():
    case = make_case(DSV3, 1, [8192], seed=51)
    topk = make_topk([8192], 1, 2048, seed=51)
    a = run_sparse(case, topk)
    b = run_sparse(case, topk)
    assert torch.equal(a, b)


def _sparse_draw(i):
    rng = np.random.default_rng(7000 + i)
    H = int(rng.choice([128, 128, 128, 8, 40]))
    n = int(rng.choice([64, 128, 192, 256]))
    v = int(rng.choice([128, 256]))
    L = int(rng.integers(1, 17))
    lens = [int(rng.integers(L, 4001)) for _ in range(int(rng.integers(1, 4)))]
    k = int(rng.integers(1, 1501))
    pad = int(rng.integers(0, 6))
    past = int(rng.integers(0, 4))
    page = int(rng.choice([0, 64]))
    dtype = torch.float32 if rng.random() < 0.2 else torch.bfloat16
    return Geometry(H=H, n=n, v=v), L, lens, k, pad, past, page, dtype


@pytest.mark.parametrize("i", range(16))
def test_random_sparse_shape(i):
    # seeded random shapes: list length (one partial tile to many), padding,
    # entries past the causal limit, ragged caches, paging, both kernel forms;
    # every element of 8 sampled heads against the oracle
    geom, L, lens, k, pad, past, page, dtype = _sparse_draw(i)
    case = make_case(geom, L, lens, dtype=dtype, seed=7100 + i, page_size=page)
    topk = make_topk(lens, L, k, seed=7200 + i, pad=pad, past_limit=past)
    got = run_sparse(case, topk)
    heads = sorted({0, geom.H - 1} | set(range(1, geom.H, max(1, geom.H // 6))))[:8]
    compare(got[:, :, heads], want_sparse(case, topk, heads=heads), dtype,
            f"sparse sweep{i} H={geom.H} n={geom.n} v={geom.v} L={L} lens={lens} k={k}")
