"""GPU parity over a seeded random sweep of call shapes.

Each case draws its geometry (n and v from the multiples of 64 up to 256,
heads from 1 to 40), its verify width L (1 to 24), batch (1 to 3), ragged
cache lengths (L to 1500, so pieces and query tiles end mid-tile), cache
layout (contiguous, pages of 64 or of 16), dtype and branch (absorbed,
materialised or the dispatcher's choice), then compares every output element
with the float64 oracle.  The shapes fall on both sides of every routing
rule (tensor-core or CUDA-core kernels, split-KV or not, one or several query
tiles and merge forms), so planning mistakes that the hand-picked cases miss
show up here.
"""

import numpy as np
import pytest
import torch

import oracle
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300 import build_lib
from mla_attention_speculative_gb300.inputs import Geometry, make_case
from parity_util import MODE_TO_ORACLE, compare, oracle_out, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 64


@pytest.fixture(scope="module", autouse=True)
def built():
    build_lib.build()
    B.lib()
    yield


def _draw(i):
    rng = np.random.default_rng(9000 + i)
    n = int(rng.choice([64, 128, 192, 256]))
    v = int(rng.choice([64, 128, 192, 256]))
    H = int(rng.choice([1, 2, 3, 5, 8, 16, 24, 33, 40]))
    L = int(rng.integers(1, 25))
    B_ = int(rng.integers(1, 4))
    lens = [int(rng.integers(L, 1501)) for _ in range(B_)]
    page = int(rng.choice([0, 0, 64, 16]))
    mode = str(rng.choice(["absorbed", "materialised", "auto"]))
    dtype = torch.float32 if rng.random() < 0.2 else torch.bfloat16
    return Geometry(H=H, n=n, v=v), L, lens, page, mode, dtype


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i):
    geom, L, lens, page, mode, dtype = _draw(i)
    case = make_case(geom, L, lens, dtype=dtype, seed=9100 + i, page_size=page)
    out, branch = run_gpu(case, mode)
    want_branch = oracle.select_branch(geom.r, geom.n, geom.v, L, lens, MODE_TO_ORACLE[mode])
    assert branch == want_branch
    what = f"sweep{i} H={geom.H} n={geom.n} v={geom.v} L={L} lens={lens} page={page} {mode}"
    compare(out, oracle_out(case), dtype, what)
