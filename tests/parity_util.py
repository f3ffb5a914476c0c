"""Helpers shared by the GPU parity tests: move a seeded case to the device,
run it through the C ABI, build the oracle's float64 inputs from the same
(dtype-rounded) values, and compare with the tolerances below.

Tolerances.  bf16 inputs with fp32 accumulation must match the float64
oracle within max-abs 2e-2 and mean-abs 2e-3 (the stated bar).  A tighter
internal gate, relative to the size of the outputs so that it bites at their
real scale, catches real mistakes: max-abs at most 2^-6 * max|want| and
relative L2 at most 1e-2.  The kernels round q_lat, the softmax weights P
and o_lat (absorbed) or the expanded K_nope/V (materialised) to bf16 for the
tensor-core contractions, and the output to bf16: each rounding carries a
relative error of at most 2^-9, which bounds the expected relative L2 error
near 3e-3 and the max-abs error near two bf16 ULPs (2 * 2^-7 relative) of the
largest output.  The configured workloads give outputs below 1 in magnitude,
where the stated absolute bar applies as written; edge cases with larger
outputs (T = 1, where the output is c_kv[0] . W_UV, or one dominant key) scale
the absolute bar by the largest |output| (S = max(1, max|want|)).
fp32 runs on CUDA cores in fp32 throughout: max-abs 1e-4*S, relative L2 1e-5.

With MLA_PARITY_LOG set to a file name, every comparison appends one JSON
line with its errors (for calibrating these bounds; the asserts are the same).
"""

from __future__ import annotations

import json
import os

import numpy as np
import torch

import oracle
from mla_attention_speculative_gb300 import binding as B
from mla_attention_speculative_gb300.inputs import Case

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
BF16_MAX_REL_GATE = 2.0 ** -6     # max-abs / max|want|
BF16_REL_L2 = 1e-2
FP32_MAX_ABS = 1e-4
FP32_REL_L2 = 1e-5

MODE_TO_ORACLE = {"auto": oracle.MODE_AUTO, "absorbed": oracle.MODE_ABSORBED,
                  "materialised": oracle.MODE_MATERIALISED}


def device_tensors(case: Case, dev="cuda"):
    t = {k: getattr(case, k).to(dev) for k in
         ("q_nope", "q_rope", "c_kv", "k_rope", "W_UK", "W_UV")}
    t["page_table"] = case.page_table.to(dev) if case.paged else None
    t["lens_dev"] = torch.tensor(case.cache_lens, dtype=torch.int32, device=dev)
    return t


def run_gpu(case: Case, mode: str, dev_t=None, **kw):
    d = dev_t if dev_t is not None else device_tensors(case)
    out, branch = B.mla_verify_attention(
        d["q_nope"], d["q_rope"], d["c_kv"], d["k_rope"], d["W_UK"], d["W_UV"],
        case.cache_lens, mode=mode, page_table=d["page_table"],
        cache_lens_dev=d["lens_dev"], **kw)
    torch.cuda.synchronize()
    B.mla_device_status()   # raises if a kernel's bounded wait ran out
    return out, branch


def oracle_inputs(case: Case):
    f = lambda x: x.float().numpy()   # exact upcast of the rounded values
    c_kv, k_rope = f(case.c_kv), f(case.k_rope)
    if case.paged:
        pt = case.page_table.numpy()
        c_kv = oracle.gather_paged(c_kv, pt, case.cache_lens, case.page_size)
        k_rope = oracle.gather_paged(k_rope, pt, case.cache_lens, case.page_size)
    return dict(q_nope=f(case.q_nope), q_rope=f(case.q_rope), c_kv=c_kv, k_rope=k_rope,
                W_UK=f(case.W_UK), W_UV=f(case.W_UV), cache_lens=case.cache_lens)


def oracle_out(case: Case, heads=None, rows=None, inputs=None):
    """The exact attention (float64); both branches equal it, so the absorbed
    form (cheaper on the CPU) serves as the expected value for either."""
    inp = inputs if inputs is not None else oracle_inputs(case)
    return oracle.absorbed(**inp, heads=heads, rows=rows)


def sample_indices(n: int, k: int, seed: int):
    rng = np.random.default_rng(seed)
    base = {0, n - 1, n // 2}
    extra = rng.choice(n, size=min(k, n), replace=False)
    return sorted(base | set(int(x) for x in extra))


def compare(got: torch.Tensor, want: np.ndarray, dtype, what=""):
    g = got.detach().float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape, (g.shape, want.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - want)
    max_abs = float(err.max())
    mean_abs = float(err.mean())
    rel = float(np.linalg.norm(g - want) / max(np.linalg.norm(want), 1e-30))
    wmax = float(np.abs(want).max())
    S = max(1.0, wmax)
    msg = (f"{what}: max_abs={max_abs:.3e} mean_abs={mean_abs:.3e} rel_l2={rel:.3e} "
           f"max|want|={wmax:.3e}")
    log = os.environ.get("MLA_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps(dict(what=what, max_abs=max_abs, mean_abs=mean_abs, rel_l2=rel,
                                    max_want=wmax, dtype=str(dtype))) + "\n")
    if dtype == torch.float32:
        assert max_abs <= FP32_MAX_ABS * S and rel <= FP32_REL_L2, msg
    else:
        assert max_abs <= BF16_MAX_ABS * S and mean_abs <= BF16_MEAN_ABS * S, msg
        assert max_abs <= BF16_MAX_REL_GATE * wmax and rel <= BF16_REL_L2, msg
    return dict(max_abs=max_abs, mean_abs=mean_abs, rel_l2=rel)
