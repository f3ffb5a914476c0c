"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases are compared element by element (several KV tiles, ragged tails,
mixed lengths, paged and packed caches, T == L).  The five measurement
configurations run at their full sizes and are compared on sampled heads and
verify rows, which the oracle computes one by one.  Branch choice is checked
exactly against the oracle's crossover.
"""

import numpy as np
import pytest
import torch

import oracle
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import (DSV3, GLM47, GLM53, Geometry, TINY,
                                                    WORKLOADS, make_case, workload_shapes)
from parity_util import (MODE_TO_ORACLE, compare, device_tensors, oracle_inputs, oracle_out,
                         run_gpu, sample_indices)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    B.lib()
    yield


def _check_branch(case, mode, branch):
    g = case.geom
    want = oracle.select_branch(g.r, g.n, g.v, case.L, case.cache_lens, MODE_TO_ORACLE[mode])
    assert branch == want, (mode, case.L, case.cache_lens, branch, want)


# ---------------------------------------------------------------------------
# Tiny fp32 layer (H=4, 512/128/128, T=512, L=4), both branches and auto
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode", ["absorbed", "materialised", "auto"])
def test_tiny_fp32_full(mode):
    w = WORKLOADS["tiny_fp32"]
    (L, lens), = workload_shapes("tiny_fp32")
    case = make_case(w["geom"], L, lens, dtype=torch.float32, seed=w["seed"])
    out, branch = run_gpu(case, mode)
    _check_branch(case, mode, branch)
    compare(out, oracle_out(case), torch.float32, f"tiny {mode}")


# ---------------------------------------------------------------------------
# Small element-by-element cases: ragged lengths, several tiles, both branches
# ---------------------------------------------------------------------------

SMALL = [
    # geometry, L, lens
    (Geometry(H=8, n=128, v=128), 1, [1]),
    (Geometry(H=8, n=128, v=128), 5, [5, 130, 1000]),
    (Geometry(H=8, n=128, v=128), 16, [16, 77, 700]),
    (Geometry(H=6, n=192, v=256), 7, [64, 65, 300]),
    (Geometry(H=4, n=256, v=256), 3, [129, 511]),
    (Geometry(H=3, n=128, v=128), 2, [2, 33]),
    (Geometry(H=128, n=128, v=128), 4, [200]),
]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("mode", ["absorbed", "materialised"])
@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_small_full(idx, mode, dtype):
    geom, L, lens = SMALL[idx]
    case = make_case(geom, L, lens, dtype=dtype, seed=100 + idx)
    out, branch = run_gpu(case, mode)
    _check_branch(case, mode, branch)
    compare(out, oracle_out(case), dtype, f"small{idx} {mode}")


@pytest.mark.parametrize("T", [1, 2, 64, 65, 200])
def test_cold_cache_T_equals_L(T):
    case = make_case(Geometry(H=8), T, [T], seed=7 + T)
    want = oracle_out(case)
    for mode in ("absorbed", "materialised", "auto"):
        out, branch = run_gpu(case, mode)
        _check_branch(case, mode, branch)
        if mode == "auto":
            assert branch == (B.BRANCH_ABSORBED if T == 1 else B.BRANCH_MATERIALISED)
        compare(out, want, torch.bfloat16, f"T=L={T} {mode}")


def test_auto_boundary_dsv3_T512():
    # 512/128/128 at T = 512: r*d*T/(r*d+(2r-d)T) = 128 exactly -> L=128 absorbed, 129 not
    for L, want in ((128, B.BRANCH_ABSORBED), (129, B.BRANCH_MATERIALISED)):
        case = make_case(Geometry(H=4), L, [512], seed=L)
        out, branch = run_gpu(case, "auto")
        assert branch == want
        heads = [0, 3]
        rows = sample_indices(L, 6, L)
        compare(out[:, rows][:, :, heads], oracle_out(case, heads=heads, rows=rows),
                torch.bfloat16, f"boundary L={L}")


def test_packed_cache_rows():
    # one [B, T, r + rope] buffer: k_rope is the tail of each row
    case = make_case(Geometry(H=8), 6, [300, 64], seed=31)
    packed = torch.cat([case.c_kv, case.k_rope], dim=-1).cuda()
    d = device_tensors(case)
    d["c_kv"] = packed[..., :512]
    d["k_rope"] = packed[..., 512:]
    want = oracle_out(case)
    for mode in ("absorbed", "materialised"):
        out, _ = run_gpu(case, mode, dev_t=d)
        compare(out, want, torch.bfloat16, f"packed {mode}")


@pytest.mark.parametrize("page", [64, 16])
def test_paged_cache_with_poisoned_tails(page):
    # rows past each sequence's length and unused pages hold NaN: they must not leak
    geom = Geometry(H=8)
    lens = [70, 64, 1, 300]
    case = make_case(geom, 1, lens, seed=41, page_size=page)
    want = oracle_out(case)
    d = device_tensors(case)
    pt = case.page_table
    poison_c = d["c_kv"].clone()
    poison_k = d["k_rope"].clone()
    used = torch.zeros(poison_c.shape[0], page, dtype=torch.bool)
    for b, T in enumerate(lens):
        for t in range(T):
            used[pt[b, t // page], t % page] = True
    poison_c[~used.cuda()] = float("nan")
    poison_k[~used.cuda()] = float("nan")
    d["c_kv"], d["k_rope"] = poison_c, poison_k
    for mode in ("absorbed", "materialised"):
        out, _ = run_gpu(case, mode, dev_t=d)
        compare(out, want, torch.bfloat16, f"paged{page} {mode}")


def test_contiguous_tail_poisoned():
    # contiguous cache with capacity beyond T: positions >= T hold NaN
    case = make_case(Geometry(H=8), 4, [100, 37], seed=43, tmax=256)
    want = oracle_out(case)
    d = device_tensors(case)
    for b, T in enumerate(case.cache_lens):
        d["c_kv"][b, T:] = float("nan")
        d["k_rope"][b, T:] = float("nan")
    for mode in ("absorbed", "materialised"):
        out, _ = run_gpu(case, mode, dev_t=d)
        compare(out, want, torch.bfloat16, f"tail {mode}")


@pytest.mark.parametrize("B,lens", [
    (32, [192] * 32),                 # pieces of exactly three KV tiles (the pipeline depth)
    (32, [130] * 32),                 # three tiles, ragged last one
    (24, [263] * 24),                 # five tiles
    (32, "mixed"),                    # pieces of 1..7 tiles across a multi-wave grid
])
def test_batched_short_pieces(B, lens):
    if lens == "mixed":
        rng = np.random.default_rng(5)
        lens = [int(x) for x in rng.integers(8, 450, size=B)]
    case = make_case(DSV3, 4, lens, seed=61, page_size=64)
    out, branch = run_gpu(case, "absorbed")
    heads = [0, 1, 64, 127]
    compare(out[:, :, heads], oracle_out(case, heads=heads), torch.bfloat16, f"short B={B}")


def test_repeat_call_is_deterministic():
    case = make_case(Geometry(H=16), 8, [1500], seed=5)
    d = device_tensors(case)
    for mode in ("absorbed", "materialised"):
        a, _ = run_gpu(case, mode, dev_t=d)
        b, _ = run_gpu(case, mode, dev_t=d)
        assert torch.equal(a, b)


# ---------------------------------------------------------------------------
# Sharp score distributions at full size: the two CTAs of an absorbed pair
# exchange their partial scores rounded to fp16, whose spacing grows with the
# score's magnitude; these cases put that rounding where it matters most
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("L", [1, 16])
def test_peaked_logits_dsv3_T8192(L):
    # queries scaled by 12: scores with a standard deviation of about 12 nats,
    # the largest about 50 nats above the mean
    case = make_case(DSV3, L, [8192], seed=200 + L, q_std=12.0)
    _sampled_check(case, ["absorbed", "materialised"], f"peaked L={L}", nheads=8, nrows=6)


@pytest.mark.parametrize("L", [1, 16])
def test_dominant_key_dsv3_T8192(L):
    # one key ahead of all others by about 65 nats, at the first position verify
    # row 0 must not see: rows l >= 1 return (nearly) its value, row 0 does not
    case = make_case(DSV3, L, [8192], seed=210 + L, dominant=30.0)
    _sampled_check(case, ["absorbed", "materialised"], f"dominant L={L}", nheads=8, nrows=6)


@pytest.mark.parametrize("geom,L,lens", [
    (Geometry(H=24), 5, [300, 1000]),      # 120 rows: one Q tile, 8 rows padding
    (GLM47, 3, [2500]),                    # 96 rows
    (Geometry(H=40), 5, [700]),            # 200 rows: second Q tile mostly padding
])
def test_nan_poisoned_workspace(geom, L, lens):
    # the workspace starts as all-ones bytes (NaN in bf16 and fp32): padded
    # query rows and any scratch read before it is written must not leak
    case = make_case(geom, L, lens, seed=220 + L)
    want = oracle_out(case)
    d = device_tensors(case)
    for mode in ("absorbed", "materialised"):
        g = B.make_geometry(geom.H, geom.r, geom.n, geom.v, geom.rope)
        need = B.mla_workspace_bytes(g, L, lens, mode)
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
        out, branch = run_gpu(case, mode, dev_t=d, workspace=ws)
        _check_branch(case, mode, branch)
        compare(out, want, torch.bfloat16, f"nan workspace {mode}")


# ---------------------------------------------------------------------------
# The measurement configurations at full size, sampled outputs
# ---------------------------------------------------------------------------

def _sampled_check(case, modes, what, nheads=6, nrows=6):
    d = device_tensors(case)
    inp = oracle_inputs(case)
    heads = sample_indices(case.geom.H, nheads, case.L)
    rows = sample_indices(case.L, nrows, case.L + 1)
    want = oracle.absorbed(**inp, heads=heads, rows=rows)
    for mode in modes:
        out, branch = run_gpu(case, mode, dev_t=d)
        _check_branch(case, mode, branch)
        compare(out[:, rows][:, :, heads], want, case.dtype, f"{what} {mode}")
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("L,lens", workload_shapes("dsv3"))
def test_dsv3_config(L, lens):
    w = WORKLOADS["dsv3"]
    case = make_case(w["geom"], L, lens, seed=w["seed"])
    modes = ["auto"] + (["materialised"] if L in (1, 16) else [])
    _sampled_check(case, modes, f"dsv3 T={lens[0]} L={L}")


@pytest.mark.parametrize("L,lens", workload_shapes("glm47_sweep"))
def test_glm47_sweep(L, lens):
    w = WORKLOADS["glm47_sweep"]
    case = make_case(w["geom"], L, lens, seed=w["seed"])
    _sampled_check(case, ["auto", "absorbed", "materialised"], f"glm L={L}")


def test_batched_paged_serving():
    w = WORKLOADS["batched_paged"]
    (L, lens), = workload_shapes("batched_paged")
    case = make_case(w["geom"], L, lens, seed=w["seed"], page_size=w["page_size"])
    _sampled_check(case, ["absorbed", "auto"], "batched paged", nheads=4, nrows=3)


@pytest.mark.parametrize("L,lens", workload_shapes("long_context"))
def test_long_context(L, lens):
    w = WORKLOADS["long_context"]
    case = make_case(w["geom"], L, lens, seed=w["seed"])
    _sampled_check(case, ["auto"], f"long L={L} T={lens[0]}", nheads=4, nrows=4)


# ---------------------------------------------------------------------------
# Which kernels run: the tensor-core path for bf16 at the supported
# geometries (contiguous and 64-row pages), the CUDA-core kernels otherwise
# ---------------------------------------------------------------------------

# absorbed: fold, attention, then the unembedding and the merge in one kernel
# (at most 64 pieces per sequence), else a merge kernel and the unembedding
TC_ABSORBED = {"fold_sm103", "absorbed_attn_sm103", "unembed_merge_sm103"}
TC_ABSORBED_MANY_PIECES = {"fold_sm103", "absorbed_attn_sm103", "merge_sm103", "unembed_sm103"}
TC_MATERIALISED = {"expand_sm103", "mat_attn_sm103"}


@pytest.mark.parametrize("mode,dtype,page,want", [
    ("absorbed", torch.bfloat16, 0, TC_ABSORBED),
    ("materialised", torch.bfloat16, 0, TC_MATERIALISED),
    ("absorbed", torch.bfloat16, 64, TC_ABSORBED),
    ("materialised", torch.bfloat16, 64, TC_MATERIALISED),
    ("materialised", torch.bfloat16, 16, {"generic_expand", "generic_materialised_attention",
                                          "generic_combine"}),
    ("materialised", torch.float32, 0, {"generic_expand", "generic_materialised_attention",
                                        "generic_combine"}),
])
def test_kernel_routing(mode, dtype, page, want):
    case = make_case(Geometry(H=8), 4, [300, 129], dtype=dtype, seed=71, page_size=page)
    B.mla_kernel_timing_enable(True)
    try:
        B.mla_kernel_timing_read(reset=True)
        out, _ = run_gpu(case, mode)
        ran = set(B.mla_kernel_timing_read(reset=True))
    finally:
        B.mla_kernel_timing_enable(False)
    assert ran == want, ran
    compare(out, oracle_out(case), dtype, f"routing {mode} page={page}")


# ---------------------------------------------------------------------------
# Failure path: a bounded device wait that runs out is reported, not hung on
# ---------------------------------------------------------------------------

def test_bounded_wait_runs_out_and_context_stays_usable():
    import ctypes
    code = ctypes.c_int32(0)
    assert B.lib().mla_device_status(ctypes.byref(code), 1) == B.MLA_OK  # start clean
    B.mla_selftest_bounded_wait()  # a barrier nothing signals: gives up after ~1 s
    assert B.lib().mla_device_status(ctypes.byref(code), 1) == B.MLA_ERR_TIMEOUT
    assert code.value == 99
    assert B.lib().mla_device_status(ctypes.byref(code), 1) == B.MLA_OK  # cleared
    assert code.value == 0
    # the context still runs a call, and that call reports no timeout
    case = make_case(Geometry(H=8), 4, [300], seed=91)
    out, _ = run_gpu(case, "absorbed")
    compare(out, oracle_out(case), torch.bfloat16, "after the self-test")


# ---------------------------------------------------------------------------
# A page id outside [0, num_pages) in the device page table: the kernels form
# no address from it, read that page's positions as zeros, and report it
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,page", [("absorbed", 64), ("materialised", 64),
                                       ("absorbed", 16)])
def test_out_of_range_page_id_is_reported(mode, page):
    case = make_case(Geometry(H=8), 2, [200, 70], seed=97, page_size=page)
    d = device_tensors(case)
    bad = d["page_table"].clone()
    bad[0, 1] = case.c_kv.shape[0] + 5       # one page of sequence 0 past the pool
    with pytest.raises(B.MlaError) as e:
        B.mla_check_page_table(bad.cpu(), case.cache_lens, page, case.c_kv.shape[0])
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    B.mla_verify_attention(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"], d["W_UK"],
                           d["W_UV"], case.cache_lens, mode=mode, page_table=bad,
                           cache_lens_dev=d["lens_dev"])
    torch.cuda.synchronize()
    with pytest.raises(B.MlaError) as e:
        B.mla_device_status()
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    assert B.mla_device_status() == 0          # the report was cleared
    out, _ = run_gpu(case, mode, dev_t=d)      # the valid table still works
    compare(out, oracle_out(case), torch.bfloat16, f"after bad page {mode}")


# ---------------------------------------------------------------------------
# Prepared call: the same entry point with its arguments marshalled once
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("mode,page", [("absorbed", 0), ("materialised", 64)])
def test_prepared_call_runs_on_new_buffer_contents(mode, page):
    case = make_case(Geometry(H=8), 4, [300, 129], seed=95, page_size=page)
    d = device_tensors(case)
    call = B.PreparedVerifyAttention(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"], d["W_UK"],
                                     d["W_UV"], case.cache_lens, mode=mode,
                                     page_table=d["page_table"], cache_lens_dev=d["lens_dev"])
    want_branch = B.BRANCH_ABSORBED if mode == "absorbed" else B.BRANCH_MATERIALISED
    assert call.run() == want_branch
    torch.cuda.synchronize()
    B.mla_device_status()
    compare(call.out, oracle_out(case), torch.bfloat16, f"prepared {mode}")
    # new queries written into the same buffers: the next run reads them
    other = make_case(Geometry(H=8), 4, [300, 129], seed=96, page_size=page)
    d["q_nope"].copy_(other.q_nope)
    d["q_rope"].copy_(other.q_rope)
    call.run()
    torch.cuda.synchronize()
    B.mla_device_status()
    case.q_nope, case.q_rope = other.q_nope, other.q_rope
    compare(call.out, oracle_out(case), torch.bfloat16, f"prepared {mode}, new queries")


@pytest.mark.parametrize("geom,L,lens,want", [
    # 76 pieces of one 64-position tile: more than the combined kernel takes
    (Geometry(H=8), 1, [76 * 64], TC_ABSORBED_MANY_PIECES),
    # 32 sequences, several sequences per unembedding CTA
    (DSV3, 8, [2048] * 32, TC_ABSORBED),
])
def test_kernel_routing_absorbed_merge_forms(geom, L, lens, want):
    case = make_case(geom, L, lens, seed=72, page_size=64)
    B.mla_kernel_timing_enable(True)
    try:
        B.mla_kernel_timing_read(reset=True)
        out, _ = run_gpu(case, "absorbed")
        ran = set(B.mla_kernel_timing_read(reset=True))
    finally:
        B.mla_kernel_timing_enable(False)
    assert ran == want, ran
    heads = [0, geom.H // 2, geom.H - 1]
    compare(out[:, :, heads], oracle_out(case, heads=heads), torch.bfloat16, f"merge forms L={L}")


@pytest.mark.parametrize("L,lens", [(1, [8192]), (16, [8192]), (32, [4096, 900]), (40, [2048])])
def test_unembed_merge_chunks(L, lens):
    # v = 256 (two column tiles per head), chunks of several verify rows, two
    # sequences of different piece counts
    case = make_case(Geometry(H=64, n=128, v=256), L, lens, seed=300 + L)
    heads = [0, 31, 63]
    rows = sample_indices(L, 4, L)
    out, _ = run_gpu(case, "absorbed")
    compare(out[:, rows][:, :, heads], oracle_out(case, heads=heads, rows=rows), torch.bfloat16,
            f"unembed-merge L={L}")


# ---------------------------------------------------------------------------
# Materialised split-KV: when the query tiles leave SMs idle the attention is
# cut into KV pieces and a combine kernel merges them
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("geom,L,lens", [
    (Geometry(H=4), 1024, [1024]),              # cold cache: the first query tiles' later pieces see nothing
    (Geometry(H=8, n=192, v=256), 1, [8192]),   # a single query row per head
    (Geometry(H=8), 130, [5000, 777]),          # two sequences, ragged
])
def test_materialised_split_kv(geom, L, lens):
    case = make_case(geom, L, lens, seed=L + len(lens))
    B.mla_kernel_timing_enable(True)
    try:
        B.mla_kernel_timing_read(reset=True)
        out, branch = run_gpu(case, "materialised")
        ran = set(B.mla_kernel_timing_read(reset=True))
    finally:
        B.mla_kernel_timing_enable(False)
    assert branch == B.BRANCH_MATERIALISED
    assert ran == TC_MATERIALISED | {"mat_combine_sm103"}, ran
    compare(out, oracle_out(case), torch.bfloat16, f"split materialised L={L} lens={lens}")
