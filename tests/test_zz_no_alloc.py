"""The entry point for callers that cannot allocate device memory.

Callers such as plugin hosts that own every device allocation, or
latency-critical loops that must not call cudaMalloc, use
mla_verify_attention_noalloc: it runs the absorbed branch with the library's
own static scratch instead of a caller-provided workspace.  These tests call
it through the C ABI and check its output against mla_verify_attention (which
uses a workspace) on two different calls in a row, so that anything the first
call leaves in the shared scratch would show up in the second.

This file is collected last on purpose, and it passes both on its own in a
fresh process and after the rest of the suite.
"""

import pytest
import torch

from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import DSV3, Geometry, make_case
from parity_util import BF16_MAX_ABS_GATE, BF16_REL_L2, device_tensors

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
    ref, br_ref = B.mla_verify_attention(*args, mode="absorbed", **kw)
    got, br = B.mla_verify_attention_noalloc(*args, **kw)
    torch.cuda.synchronize()
    assert br == br_ref == B.BRANCH_ABSORBED
    return got.float(), ref.float()


def _close(got, ref):
    err = (got - ref).abs()
    scale = max(1.0, float(ref.abs().max()))
    rel = float(torch.linalg.norm(got - ref) / torch.linalg.norm(ref))
    assert float(err.max()) <= BF16_MAX_ABS_GATE * scale and rel <= BF16_REL_L2, \
        (float(err.max()), rel)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    first = make_case(DSV3, 16, [8192], seed=77)
    second = make_case(Geometry(H=32), 4, [3001, 700], seed=78)   # smaller, different shape
    for case in (first, second):
        got, ref = _both(case)
        _close(got, ref)


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
