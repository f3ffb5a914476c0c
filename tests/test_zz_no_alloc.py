"""The entry point for callers that cannot allocate device memory.

Callers such as plugin hosts that own every device allocation, or
latency-critical loops that must not call cudaMalloc, use
mla_verify_attention_noalloc: it runs the absorbed branch with the library's
own static scratch instead of a caller-provided workspace.  These tests call
it through the C ABI and check that its output is bit for bit the output of
mla_verify_attention (which uses a workspace and the same kernels and plan),
over several different calls in a row: a large call first, then calls whose
query rows do not fill whole 128-row tiles (padding rows read whatever the
previous call left in the shared scratch) and a paged cache, so anything a
call leaves behind would show up in the next.  One call is also compared with
the float64 oracle.

This file is collected last on purpose, and it passes both on its own in a
fresh process and after the rest of the suite.
"""

import pytest
import torch

from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import DSV3, Geometry, make_case
from parity_util import compare, device_tensors, oracle_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    B.lib()
    yield


def _both(case):
    d = device_tensors(case)
    args = (d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"], d["W_UK"], d["W_UV"],
            case.cache_lens)
    kw = dict(page_table=d["page_table"], cache_lens_dev=d["lens_dev"])
    got, br = B.mla_verify_attention_noalloc(*args, **kw)
    torch.cuda.synchronize()
    ref, br_ref = B.mla_verify_attention(*args, mode="absorbed", **kw)
    torch.cuda.synchronize()
    B.mla_device_status()
    assert br == br_ref == B.BRANCH_ABSORBED
    return got, ref


CALLS = [
    (DSV3, 16, [8192], 0),                 # 2048 query rows: most of the scratch in use
    (Geometry(H=32), 1, [3001, 700], 0),   # 32 rows per sequence: 96 padding rows per tile
    (Geometry(H=8), 3, [70, 200, 3], 64),  # paged cache, 24 rows per sequence
    (Geometry(H=40), 5, [700], 0),         # 200 rows: a second, mostly padding, tile
]


def test_noalloc_matches_workspace_entry_point_call_after_call():
    for i, (geom, L, lens, page) in enumerate(CALLS):
        case = make_case(geom, L, lens, seed=77 + i, page_size=page)
        got, ref = _both(case)
        assert torch.equal(got, ref), f"call {i}: noalloc differs from the workspace call"
        if i == 1:
            compare(got, oracle_out(case), torch.bfloat16, "noalloc vs oracle")


def test_noalloc_rejects_calls_beyond_static_scratch():
    # 32 sequences of 8 rows at H=128 need more than the 32 MiB of static scratch
    case = make_case(DSV3, 8, [2048] * 32, seed=79)
    d = device_tensors(case)
    with pytest.raises(B.MlaError) as e:
        B.mla_verify_attention_noalloc(d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"],
                                       d["W_UK"], d["W_UV"], case.cache_lens,
                                       cache_lens_dev=d["lens_dev"])
    assert e.value.status == B.MLA_ERR_WORKSPACE
    assert "static scratch" in str(e.value)
