"""C-ABI checks that need no GPU: the library loads, exports every entry point
the header declares, and its host logic (crossover, branch choice, workspace
plan, argument validation) behaves.  No compute call is made here."""

import ctypes
import os
import re

import pytest

import oracle
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300.inputs import WORKLOADS, workload_shapes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    yield


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(mla_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_entry_points():
    d = _declared()
    for must in ("mla_max_absorbed_queries", "mla_select_branch", "mla_workspace_bytes",
                 "mla_verify_attention", "mla_status_string", "mla_last_error"):
        assert must in d


@pytest.mark.parametrize("name", _declared())
def test_library_exports_declared_symbol(name):
    lib = ctypes.CDLL(B.LIB_PATH)
    assert hasattr(lib, name), name


def test_threshold_matches_oracle_grid():
    for r in (64, 256, 512, 1024):
        for n in (16, 64, 128, 192, 256):
            for v in (16, 64, 128, 256):
                for T in (0, 1, 2, 3, 17, 512, 2048, 8192, 131072, 1 << 31):
                    want = oracle.max_absorbed_queries(r, n, v, T if T > 0 else None)
                    assert B.mla_max_absorbed_queries(r, n, v, T) == want, (r, n, v, T)


def test_threshold_printed_values_through_abi():
    assert B.mla_max_absorbed_queries(512, 128, 128) == 170
    assert B.mla_max_absorbed_queries(512, 192, 256) == 398
    assert B.mla_max_absorbed_queries(512, 256, 256) == 512
    assert B.mla_max_absorbed_queries(512, 192, 256, 8192) == 379
    assert B.mla_max_absorbed_queries(0, 128, 128) == -1


def test_batch_threshold_matches_oracle():
    lens_sets = [[1024, 32768, 5000], [8192] * 4, [77], list(range(1000, 33000, 1000))]
    for lens in lens_sets:
        for geom in ((512, 128, 128), (512, 192, 256), (512, 256, 256)):
            assert B.mla_max_absorbed_queries_batch(*geom, lens) == \
                oracle.max_absorbed_queries_batch(*geom, lens)
    assert B.mla_max_absorbed_queries_batch(512, 128, 128, [0]) == -1


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_branch_choice_matches_oracle_on_workloads(name):
    w = WORKLOADS[name]
    g = w["geom"]
    geom = B.make_geometry(g.H, g.r, g.n, g.v, g.rope, w["dtype"])
    for L, lens in workload_shapes(name):
        for mode, m in (("auto", oracle.MODE_AUTO), ("absorbed", oracle.MODE_ABSORBED),
                        ("materialised", oracle.MODE_MATERIALISED)):
            assert B.mla_select_branch(geom, L, lens, mode) == \
                oracle.select_branch(g.r, g.n, g.v, L, lens, m), (name, L, mode)


def test_glm_sweep_branches_flip_between_379_and_398():
    import torch
    geom = B.make_geometry(32, 512, 192, 256, 64, torch.bfloat16)
    assert B.mla_select_branch(geom, 379, [8192]) == B.BRANCH_ABSORBED
    assert B.mla_select_branch(geom, 380, [8192]) == B.BRANCH_MATERIALISED
    assert B.mla_select_branch(geom, 398, [8192]) == B.BRANCH_MATERIALISED


def test_workspace_bytes_positive_and_branch_dependent():
    import torch
    geom = B.make_geometry(128, 512, 128, 128, 64, torch.bfloat16)
    a = B.mla_workspace_bytes(geom, 4, [8192], "absorbed")
    m = B.mla_workspace_bytes(geom, 4, [8192], "materialised")
    assert a > 0 and m > 0
    # the materialised branch holds the expanded K_nope/V: T*H*(n+v)*2 bytes at least
    assert m >= 8192 * 128 * 256 * 2


def _geom(**kw):
    import torch
    base = dict(H=4, r=512, n=128, v=128, rope=64, dtype=torch.bfloat16)
    base.update(kw)
    return B.make_geometry(base["H"], base["r"], base["n"], base["v"], base["rope"],
                           base["dtype"])


@pytest.mark.parametrize("kw,L,lens", [
    (dict(), 5, [4]),            # L > T
    (dict(), 0, [4]),            # L < 1
    (dict(H=0), 1, [4]),         # no heads
    (dict(r=500), 1, [4]),       # row not a whole number of 16-byte vectors
    (dict(n=-8), 1, [4]),
])
def test_invalid_geometry_and_lengths(kw, L, lens):
    with pytest.raises(B.MlaError) as e:
        B.mla_workspace_bytes(_geom(**kw), L, lens)
    assert e.value.status == B.MLA_ERR_INVALID_ARG


def _call(**over):
    """Raw C call with fake (never dereferenced) device pointers; returns the status.

    Every case below fails validation, which happens before any launch, so no
    CUDA call is made."""
    lib = B.lib()
    geom = _geom()
    lens = (ctypes.c_int32 * 1)(64)
    fake = 0x10000
    args = dict(q_nope=fake, q_rope=fake, c_kv=fake, k_rope=fake, cs=512, ks=64, seq=64,
                W_UK=fake, W_UV=fake, lens_dev=fake, lens_host=lens, batch=1, L=4,
                page_table=None, page_size=0, max_pages=0, num_pages=0, mode=0, out=fake,
                ws=None, ws_bytes=0, stream=None)
    args.update(over)
    branch = ctypes.c_int32(0)
    return lib.mla_verify_attention(
        ctypes.byref(geom), args["q_nope"], args["q_rope"], args["c_kv"], args["k_rope"],
        args["cs"], args["ks"], args["seq"], args["W_UK"], args["W_UV"], args["lens_dev"],
        args["lens_host"], args["batch"], args["L"], args["page_table"], args["page_size"],
        args["max_pages"], args["num_pages"], args["mode"], args["out"], args["ws"],
        args["ws_bytes"], args["stream"], ctypes.byref(branch))


@pytest.mark.parametrize("over,status", [
    (dict(q_nope=None), B.MLA_ERR_INVALID_ARG),
    (dict(out=None), B.MLA_ERR_INVALID_ARG),
    (dict(c_kv=0x10008), B.MLA_ERR_INVALID_ARG),          # misaligned
    (dict(cs=100), B.MLA_ERR_INVALID_ARG),                # stride below r
    (dict(L=65), B.MLA_ERR_INVALID_ARG),                  # L > T
    (dict(mode=7), B.MLA_ERR_INVALID_ARG),
    (dict(batch=0), B.MLA_ERR_INVALID_ARG),
    (dict(page_table=0x20000, page_size=64, max_pages=0, num_pages=4), B.MLA_ERR_INVALID_ARG),
    (dict(page_table=0x20000, page_size=16, max_pages=2, num_pages=4), B.MLA_ERR_INVALID_ARG),
    (dict(), B.MLA_ERR_WORKSPACE),                        # no workspace given
    (dict(ws=0x30000, ws_bytes=16), B.MLA_ERR_WORKSPACE),
])
def test_verify_attention_rejects_before_launch(over, status):
    assert _call(**over) == status
    assert B.mla_last_error() != ""


def test_status_strings():
    assert B.status_string(0) == "MLA_OK"
    assert B.status_string(-3) == "MLA_ERR_WORKSPACE"
    assert B.status_string(-99) == "MLA_ERR_UNKNOWN"


# ---------------------------------------------------------------------------
# Host-side page-table validation
# ---------------------------------------------------------------------------

def test_page_table_check_accepts_valid_table():
    table = [[3, 0, 7], [1, 2, -1]]          # -1 past sequence 1's last page is not read
    B.mla_check_page_table(table, [130, 100], 64, 8)


@pytest.mark.parametrize("table,lens,num_pages,bad", [
    ([[3, 8, 0]], [130], 8, "page_table[0][1] = 8"),     # one past the pool
    ([[0, -1]], [65], 4, "page_table[0][1] = -1"),       # negative id inside the sequence
    ([[0, 1], [2, 99]], [10, 128], 4, "page_table[1][1] = 99"),
    ([[0, 1]], [129], 4, "needs 3 pages"),               # table too narrow for T
])
def test_page_table_check_rejects_out_of_range(table, lens, num_pages, bad):
    with pytest.raises(B.MlaError) as e:
        B.mla_check_page_table(table, lens, 64, num_pages)
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    assert bad in str(e.value)


def test_noalloc_binding_rejects_non_contiguous_views():
    # the tensor maps assume row-major operands: a transposed view must be
    # refused before anything reaches the library
    import torch
    q = torch.zeros(1, 2, 4, 128, dtype=torch.bfloat16).transpose(1, 2)
    qr = torch.zeros(1, 4, 2, 64, dtype=torch.bfloat16)
    ckv = torch.zeros(1, 64, 512, dtype=torch.bfloat16)
    kr = torch.zeros(1, 64, 64, dtype=torch.bfloat16)
    wuk = torch.zeros(2, 128, 512, dtype=torch.bfloat16)
    wuv = torch.zeros(2, 512, 128, dtype=torch.bfloat16)
    for fn in (B.mla_verify_attention_noalloc, B.mla_verify_attention):
        with pytest.raises(ValueError, match="q_nope must be contiguous"):
            fn(q, qr, ckv, kr, wuk, wuv, [64])


# ---------------------------------------------------------------------------
# Sparse (top-k) entry points: host-side checks, no GPU
# ---------------------------------------------------------------------------

def _sparse_call(topk=0x40000, k=8, **over):
    lib = B.lib()
    geom = _geom()
    lens = (ctypes.c_int32 * 1)(64)
    fake = 0x10000
    a = dict(q_nope=fake, L=4, ws=None, ws_bytes=0)
    a.update(over)
    return lib.mla_verify_attention_sparse(
        ctypes.byref(geom), a["q_nope"], fake, fake, fake, 512, 64, 64, fake, fake, fake, lens,
        1, a["L"], topk, k, None, 0, 0, 0, fake, a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("over,status", [
    (dict(topk=None), B.MLA_ERR_INVALID_ARG),
    (dict(k=0), B.MLA_ERR_INVALID_ARG),
    (dict(topk=0x40004), B.MLA_ERR_INVALID_ARG),   # misaligned list
    (dict(L=65), B.MLA_ERR_INVALID_ARG),           # L > T
    (dict(), B.MLA_ERR_WORKSPACE),                 # no workspace given
])
def test_sparse_call_rejects_before_launch(over, status):
    assert _sparse_call(**over) == status
    assert B.mla_last_error() != ""


def test_sparse_workspace_follows_the_list_length():
    g = _geom(H=128)
    small = B.mla_sparse_workspace_bytes(g, 1, [32768], 64)
    large = B.mla_sparse_workspace_bytes(g, 1, [32768], 2048)
    dense = B.mla_workspace_bytes(g, 1, [32768], "absorbed")
    assert 0 < small <= large <= dense


def test_batch_beyond_grid_limit_is_rejected():
    lens = [64] * 65536
    with pytest.raises(B.MlaError) as e:
        B.mla_workspace_bytes(_geom(), 1, lens)
    assert e.value.status == B.MLA_ERR_INVALID_ARG
    assert "65535" in str(e.value)


@pytest.mark.parametrize("kw", [dict(dim=48), dict(dim=1024), dict(new_tokens=0),
                                dict(cache_len=3, new_tokens=4), dict(cap=10)])
def test_indexer_pool_update_rejects_bad_arguments(kw):
    args = dict(dim=128, cache_len=100, new_tokens=4, cap=25)
    args.update(kw)
    st = B.IndexerPoolState()
    lib = B.lib()
    status = lib.mla_indexer_pool_update(0x10000, 0, args["dim"], 1 << 20, 1, args["dim"],
                                         args["cache_len"], args["new_tokens"], 0, 0x20000,
                                         args["cap"], ctypes.byref(st), None, None)
    assert status == B.MLA_ERR_INVALID_ARG
    assert st.length == -1          # the state is untouched by a rejected call


@pytest.mark.parametrize("kw,status", [
    (dict(), B.MLA_ERR_WORKSPACE),                      # valid, but no workspace given
    (dict(q=0x10004), B.MLA_ERR_INVALID_ARG),           # q not 16-byte aligned
    (dict(pooled=0x20008), B.MLA_ERR_INVALID_ARG),      # pooled not 16-byte aligned
    (dict(new_tokens=33), B.MLA_ERR_INVALID_ARG),
    (dict(dim=512, new_tokens=32), B.MLA_ERR_INVALID_ARG),   # 64 KB of queries > 48 KB
    (dict(cap=10), B.MLA_ERR_INVALID_ARG),
    (dict(k=0), B.MLA_ERR_INVALID_ARG),
])
def test_indexer_select_rejects_before_launch(kw, status):
    a = dict(q=0x10000, pooled=0x20000, cap=25, dim=128, cache_len=100, new_tokens=4, k=8)
    a.update(kw)
    st = B.lib().mla_indexer_select(a["q"], a["pooled"], a["cap"], 1, a["dim"], a["cache_len"],
                                    a["new_tokens"], a["k"], None, 0x30000, None, 0, None)
    assert st == status
    assert B.mla_last_error() != ""
