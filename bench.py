#!/usr/bin/env python
"""MLA verify benchmark: layer-calls/s and us/call at cache 8K, L = 1..16.

Workload (DeepSeek-V3-like geometry): H=128 heads, latent r=512, nope n=128,
value v=128, RoPE 64, bf16 with fp32 accumulation, one sequence of cache
length T=8192 (each layer's c_kv and k_rope packed as [T, 576] rows),
verify widths L in {1, 2, 4, 8, 16}, crossover dispatch ("auto", which picks
the absorbed branch at every one of these widths).  One step is one verify
call per width (5 layer-calls).  Each call uses its own layer's weights and
cache; ten layers rotate (about 430 MB, larger than the 129 MB L2), so every
call streams its operands from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  Under torchrun every rank runs the same
replica (no data exchange); value is the calls of all ranks over the slowest
rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WIDTHS = (1, 2, 4, 8, 16)
CACHE_LEN = 8192
NUM_LAYERS = 10
METRIC = "MLA verify layer-calls/s (cache 8K, L=1..16)"
UNIT = "calls/s"
WORKLOAD = "dsv3-like B=1 T=8192 L=1,2,4,8,16 auto-dispatch (absorbed)"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shapes", "--no-materialised", dest="no_shapes", action="store_true",
                    help="skip the secondary shapes (crossover sweep, batched paged, long "
                         "context, materialised)")
    ap.add_argument("--shape-groups", default=None,
                    help="comma-separated names of the secondary shape groups to run (default "
                         "all: crossover_glm47_T8192, batched_paged, long_context, "
                         "dsv3_forced_materialised, sparse_dsv3_k2048, draft_cap_dsv3_T8192, "
                         "indexer_pool_T131072, sparse_step_dsv3_T32768, conv_snapshots_H8192)")
    ap.add_argument("--widths", default=None,
                    help="comma-separated verify widths instead of 1,2,4,8,16 (for profiling "
                         "one width; the line then describes that workload, not the headline)")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest of every rank's x (a host float), through one all-reduce on
    `device` (the GPU for NCCL, the CPU for gloo); x itself on one rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, seconds_slowest):
    """Whole-job throughput of independent replicas: the units every rank
    processed over the slowest rank's time."""
    return world * units_per_rank / seconds_slowest


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# Algorithmic work per kernel launch (bytes that must cross HBM, flops that
# the method must do), for the roofline of the dominant kernel.
# ---------------------------------------------------------------------------

def visible(L: int, T: int) -> int:
    """Positions the L verify rows of one sequence see together: row l sees
    t <= T - L + l, so L (T - L) + L (L + 1) / 2 in all (causal work only)."""
    return L * (T - L) + L * (L + 1) // 2


def kernel_work(kernel: str, geom, L: int, lens, topk_k: int = 0):
    """(bytes, flops) one launch of `kernel` must move / do for one call.

    Bytes count what the kernel's role needs to cross HBM once, with bf16
    intermediates (q_lat, o_lat, the expanded K/V) as the minimal hand-off
    between kernels; split-KV partials are an implementation cost and are not
    counted.  Flops count the contraction the kernel performs over the
    positions each row may see (2 per multiply-add; masked work not counted).
    A sparse call (topk_k > 0) reads topk_k listed rows per verify row."""
    bf = 2
    H, r, n, v, rope = geom.H, geom.r, geom.n, geom.v, geom.rope
    d = n + v
    B = len(lens)
    rows = B * L * H
    sT = sum(lens)
    vis = sum(visible(L, T) for T in lens)
    cache = sT * (r + rope) * bf
    if topk_k:
        vis = B * L * topk_k
        cache = vis * (r + rope) * bf
    fold = (H * n * r * bf + rows * (n + r) * bf, 2 * rows * n * r)
    attend = (cache + rows * (r + rope) * bf + rows * r * bf, 2 * H * vis * (2 * r + rope))
    unembed = (H * r * v * bf + rows * (r + v) * bf, 2 * rows * r * v)
    expand = (sT * r * bf + H * r * d * bf + sT * H * d * bf, 2 * sT * r * H * d)
    mat_attn = (sT * H * d * bf + sT * rope * bf + rows * (n + rope + v) * bf,
                2 * H * (n + rope + v) * vis)
    table = {
        "fold_sm103": fold, "generic_fold": fold,
        "absorbed_attn_sm103": attend, "generic_absorbed_attention": attend,
        "absorbed_attn_sparse_sm103": attend,
        "unembed_merge_sm103": unembed, "unembed_sm103": unembed,
        "generic_combine_unembed": unembed,
        "expand_sm103": expand, "generic_expand": expand,
        "mat_attn_sm103": mat_attn, "generic_materialised_attention": mat_attn,
    }
    return table.get(kernel)


def _work(kernel: str, L: int, T: int):
    """kernel_work for the headline workload (DSV3-like, one sequence)."""
    from mla_attention_speculative_gb300.inputs import DSV3
    return kernel_work(kernel, DSV3, L, [T])


def call_work(branch: str, geom, L: int, lens, topk_k: int = 0):
    """Algorithmic (bytes, flops, cache_bytes) of one verify call, as the
    method must do it (masked positions and the softmax not counted;
    vis_b = visible(L, T_b)):
      absorbed:     flops = sum_b 2 H (L n r + vis_b (r + rope) + vis_b r + L r v)
                    bytes = sum_b T_b (r + rope) 2 + H (n r + r v) 2 + B L H (n + rope + v) 2
      materialised: flops = sum_b 2 H (T_b r d + vis_b (n + rope) + vis_b v)
                    bytes = the absorbed bytes + 2 sum_b T_b H d 2 (the expanded
                    keys and values written once and read once)."""
    H, r, n, v, rope = geom.H, geom.r, geom.n, geom.v, geom.rope
    d = n + v
    B = len(lens)
    cache = sum(T * (r + rope) * 2 for T in lens)
    if topk_k:  # sparse: every verify row reads its topk_k listed rows
        cache = B * L * topk_k * (r + rope) * 2
    byts = cache + H * (n * r + r * v) * 2 + B * L * H * (n + rope + v) * 2
    if topk_k:
        flops = B * 2 * H * L * (n * r + topk_k * (2 * r + rope) + r * v)
    elif branch == "absorbed":
        flops = sum(2 * H * (L * n * r + visible(L, T) * (2 * r + rope) + L * r * v)
                    for T in lens)
    else:
        flops = sum(2 * H * (T * r * d + visible(L, T) * (n + rope + v)) for T in lens)
        byts += 2 * sum(T * H * d * 2 for T in lens)
    return byts, flops, cache


def call_roofline(branch: str, geom, L: int, lens, us: float, peaks, topk_k: int = 0) -> dict:
    """Fraction of the call roofline max(bytes / BW, flops / peak) reached in `us`."""
    byts, flops, cache = call_work(branch, geom, L, lens, topk_k)
    t_b = byts / (peaks["hbm_gbs"] * 1e3)      # us
    t_f = flops / (peaks["bf16_tflops"] * 1e6)  # us
    t_c = cache / (peaks["hbm_gbs"] * 1e3)
    return {"us": us, "roofline_us": max(t_b, t_f), "bound": "hbm" if t_b >= t_f else "tensor",
            "frac": max(t_b, t_f) / us, "cache_only_frac": max(t_c, t_f) / us}


def kernel_rates(kernel: str, geom, L: int, lens, us: float, peaks, topk_k: int = 0) -> dict:
    """A launch's achieved HBM and tensor rates and the fraction of the bound
    that its algorithmic work puts it under."""
    w = kernel_work(kernel, geom, L, lens, topk_k)
    ent = {"us": us}
    if w is None:
        return ent
    gbs = w[0] / (us * 1e-6) / 1e9
    tfs = w[1] / (us * 1e-6) / 1e12
    t_b, t_f = w[0] / (peaks["hbm_gbs"] * 1e9), w[1] / (peaks["bf16_tflops"] * 1e12)
    ent.update(gbs=gbs, hbm_frac=gbs / peaks["hbm_gbs"], tflops=tfs,
               tensor_frac=tfs / peaks["bf16_tflops"], bound="hbm" if t_b >= t_f else "tensor")
    ent["frac"] = ent["hbm_frac"] if t_b >= t_f else ent["tensor_frac"]
    return ent


# Secondary measurements beside the headline (each its own workload, its own
# line in the "shapes" object):
# - the GLM-4.7-Flash-like crossover sweep at cache 8192 with each branch
#   forced (the pages time both branches across L to validate the formula);
# - the batched paged serving verify (32 sequences, T ~ U{1024..32768}, L = 8,
#   page 64, shuffled page table, absorbed);
# - long-context verify (512/256/256, H = 64, B = 4, T = 131072, L = 1, 5, 8,
#   16, auto) and its cold prefill (T = L = 2048, auto -> materialised);
# - the DeepSeek-V3-like width-16 call forced onto the materialised branch;
# - the sparse (top-k) call at the sparse model's budget of 2048 positions
#   (DeepSeek-V3-like geometry, seeded random lists) at caches of 8K and 32K.
CROSSOVER_L = (1, 16, 64, 128, 256, 379, 398, 512, 1024, 2048)
L2_ROTATE_BYTES = 256 << 20   # rotate input copies until a graph touches this much


def _shape_list():
    from mla_attention_speculative_gb300 import inputs as I
    out = []
    for L in CROSSOVER_L:
        for mode in ("absorbed", "materialised"):
            out.append(dict(group="crossover_glm47_T8192", geom=I.GLM47, L=L, lens=[8192],
                            mode=mode, page=0))
    out.append(dict(group="batched_paged", geom=I.DSV3, L=8,
                    lens=I.workload_shapes("batched_paged")[0][1], mode="absorbed", page=64))
    for L, lens in I.workload_shapes("long_context"):
        out.append(dict(group="long_context", geom=I.GLM53, L=L, lens=lens, mode="auto", page=0))
    out.append(dict(group="dsv3_forced_materialised", geom=I.DSV3, L=16, lens=[8192],
                    mode="materialised", page=0))
    for T, L in ((8192, 1), (32768, 1), (32768, 4), (32768, 8)):
        out.append(dict(group="sparse_dsv3_k2048", geom=I.DSV3, L=L, lens=[T], mode="sparse",
                        page=0, topk=2048))
    for L in range(1, DRAFT_CAP_MAX + 2):
        out.append(dict(group="draft_cap_dsv3_T8192", geom=I.DSV3, L=L, lens=[8192],
                        mode="auto", page=0))
    return out


DRAFT_CAP_MAX = 16
DRAFT_P = (0.5, 0.7, 0.8, 0.9)


def _draft_caps(B, group):
    """The draft cap that "Draft caps and calibration" picks from a measured
    verify curve: verify(w) is this build's µs per layer call over w rows
    (w = 1 .. DRAFT_CAP_MAX + 1, a cap C verifying C + 1 rows), for a few
    acceptance rates p, with the drafter free and at a tenth of one verify."""
    us = {e["L"]: e["us_per_call"] for e in group["calls"]}
    curve = [us[w] for w in range(1, DRAFT_CAP_MAX + 2)]
    caps = []
    for p in DRAFT_P:
        for drafter in (0.0, 0.1 * curve[0]):
            cap, speedup = B.mla_select_draft_cap(p, curve, drafter, DRAFT_CAP_MAX)
            caps.append({"p": p, "drafter_us": drafter, "cap": cap,
                         "speedup": speedup[cap]})
    return {"verify_us": curve, "caps": caps}


def _bench_shapes(B, dev, peaks, reps, only=None):
    """Per shape: us per call (CUDA graph of calls over rotating input copies so
    the working set exceeds L2, CUDA events), the call roofline, and each
    kernel's achieved rates (events around each launch, eager calls)."""
    import torch
    from mla_attention_speculative_gb300 import inputs as I
    groups = {}
    for k, sh in enumerate(_shape_list()):
        if only is not None and sh["group"] not in only:
            continue
        geom, L, lens, mode, page = sh["geom"], sh["L"], sh["lens"], sh["mode"], sh["page"]
        kk = sh.get("topk", 0)
        layer_bytes = (sum(lens) * (geom.r + geom.rope)
                       + geom.H * geom.r * (geom.n + geom.v)) * 2
        copies = max(1, min(8, -(-L2_ROTATE_BYTES // layer_bytes)))
        cases = [I.make_case(geom, L, lens, seed=3000 + 17 * k + i, page_size=page, device=dev)
                 for i in range(copies)]
        lens_dev = torch.tensor(lens, dtype=torch.int32, device=dev)
        g = B.make_geometry(geom.H, geom.r, geom.n, geom.v, geom.rope, torch.bfloat16)
        if kk:
            ws = B.new_workspace(B.mla_sparse_workspace_bytes(g, L, lens, kk), dev)
            lists = [I.make_topk(lens, L, kk, seed=4000 + i, device=dev) for i in range(copies)]
        else:
            ws = B.new_workspace(B.mla_workspace_bytes(g, L, lens, mode), dev)
        out = torch.empty((len(lens), L, geom.H, geom.v), dtype=torch.bfloat16, device=dev)
        br = {}

        def call(i):
            c = cases[i]
            if kk:
                B.mla_verify_attention_sparse(
                    c.q_nope, c.q_rope, c.c_kv, c.k_rope, c.W_UK, c.W_UV, lens,
                    lists[i], out=out, workspace=ws, cache_lens_dev=lens_dev)
                br["b"] = B.BRANCH_ABSORBED
                return
            _, br["b"] = B.mla_verify_attention(
                c.q_nope, c.q_rope, c.c_kv, c.k_rope, c.W_UK, c.W_UV, lens, mode=mode,
                out=out, workspace=ws, cache_lens_dev=lens_dev,
                page_table=c.page_table if page else None)

        for i in range(copies):
            call(i)
        torch.cuda.synchronize()
        st = torch.cuda.Stream(dev)
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=st):
            for i in range(copies):
                call(i)
        gr.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            gr.replay()
        b.record()
        torch.cuda.synchronize()
        us_call = a.elapsed_time(b) * 1e3 / (reps * copies)
        B.mla_kernel_timing_read(reset=True)
        B.mla_kernel_timing_enable(True)
        for _ in range(max(1, reps // 2)):
            for i in range(copies):
                call(i)
        torch.cuda.synchronize()
        B.mla_kernel_timing_enable(False)
        kt = B.mla_kernel_timing_read(reset=True)
        branch = B.BRANCH_NAMES[br["b"]]
        ent = {"L": L, "mode": mode, "branch": branch, "us_per_call": us_call,
               "call_roofline": call_roofline(branch, geom, L, lens, us_call, peaks, kk),
               "kernels": {kn: kernel_rates(kn, geom, L, lens, ms * 1e3 / max(nl, 1), peaks, kk)
                           for kn, (nl, ms) in kt.items()}}
        if kk:
            ent["topk"] = kk
        if len(lens) > 1:
            ent["B"] = len(lens)
            ent["sum_T"] = sum(lens)
        else:
            ent["T"] = lens[0]
        if page:
            ent["page_size"] = page
        gd = groups.setdefault(sh["group"], {
            "geometry": f"H={geom.H} r={geom.r} n={geom.n} v={geom.v} rope={geom.rope}",
            "calls": []})
        gd["calls"].append(ent)
        del cases, ws, out, gr
        torch.cuda.empty_cache()
    cx = groups.get("crossover_glm47_T8192")
    if cx:
        from mla_attention_speculative_gb300.inputs import GLM47
        t = {}
        for e in cx["calls"]:
            t.setdefault(e["L"], {})[e["mode"]] = e["us_per_call"]
        first = next((L for L in sorted(t) if t[L]["materialised"] < t[L]["absorbed"]), None)
        cx["formula_threshold"] = B.mla_max_absorbed_queries(GLM47.r, GLM47.n, GLM47.v, 8192)
        cx["measured_crossover"] = {
            "first_L_materialised_faster": first,
            "us": {str(L): {"absorbed": v["absorbed"], "materialised": v["materialised"]}
                   for L, v in sorted(t.items())}}
    dc = groups.get("draft_cap_dsv3_T8192")
    if dc:
        dc["draft_cap"] = _draft_caps(B, dc)
    if only is None or "indexer_pool_T131072" in only:
        groups["indexer_pool_T131072"] = _bench_indexer(B, dev, peaks, reps)
    if only is None or "sparse_step_dsv3_T32768" in only:
        groups["sparse_step_dsv3_T32768"] = _bench_sparse_step(B, dev, reps)
    if only is None or "conv_snapshots_H8192" in only:
        groups["conv_snapshots_H8192"] = _bench_snapshots(B, dev, peaks, reps)
    return {"groups": groups, "peak_tflops": peaks["bf16_tflops"], "peak_gbs": peaks["hbm_gbs"],
            "peak_source": f"of {peaks['source']}",
            "timing": "CUDA graph of one call per input copy, copies rotated until the "
                      "working set exceeds 256 MB (> L2); work counts causal positions only"}


def _bench_indexer(B, dev, peaks, reps):
    """The sparse model's indexer step at a 128K cache: a full pool of the
    windows of four, the incremental (tail-only) step for S = 1, 4, 8 new
    tokens, and the top-512-window selection for 8 new tokens.  Device time
    per launch from events around each launch; six key buffers rotate so a
    full pool reads its keys from HBM."""
    import torch
    T, d, k = 131072, 128, 512
    W = T // 4
    copies = 6
    g = torch.Generator(device=dev).manual_seed(5000)
    keys = [torch.randn(1, T, d, generator=g, device=dev).to(torch.bfloat16) for _ in range(copies)]
    pooled = [torch.zeros((1, W, d), device=dev) for _ in range(copies)]
    q = torch.randn(1, 8, d, generator=g, device=dev)
    out = {"geometry": f"keys bf16 [1, {T}, {d}], windows of four, k = {k} windows", "calls": []}

    def timed(fn, n):
        B.mla_kernel_timing_read(reset=True)
        B.mla_kernel_timing_enable(True)
        for i in range(n):
            fn(i)
        torch.cuda.synchronize()
        B.mla_kernel_timing_enable(False)
        return B.mla_kernel_timing_read(reset=True)

    n = max(6, reps)
    for S in (T, 1, 4, 8):
        def step(i, S=S):
            st = B.IndexerPoolState()
            if S != T:   # a pool that remembers the cache before this step
                st.length, st.batch, st.dim = T - S, 1, d
            B.mla_indexer_pool_update(keys[i % copies], T, S, pooled[i % copies], st)
        step(0)
        kt = timed(step, n)
        nl, ms = kt["indexer_pool_windows"]
        us = ms * 1e3 / nl
        ent = {"step": "full pool" if S == T else f"incremental, S = {S}", "us": us}
        if S == T:
            byts = T * d * 2 + W * d * 4
            ent.update(gbs=byts / (us * 1e-6) / 1e9, hbm_frac=byts / (us * 1e-6) / 1e9 /
                       peaks["hbm_gbs"], bound="hbm")
        out["calls"].append(ent)
    B.mla_indexer_select(q, pooled[0], T, k)
    kt = timed(lambda i: B.mla_indexer_select(q, pooled[i % copies], T, k), n)
    sel = {"step": "select top-512 windows, S = 8"}
    for name, (nl, ms) in kt.items():
        sel[name + "_us"] = ms * 1e3 / nl
    byts = W * d * 4 + 8 * W * 4
    sel["score_gbs"] = byts / (sel["indexer_score_windows_us"] * 1e-6) / 1e9
    sel["score_hbm_frac"] = sel["score_gbs"] / peaks["hbm_gbs"]
    # the whole call (scoring, then the selection chained to it): a CUDA graph
    # of calls over the rotating pools, events around its replays
    ncall = 2 * copies
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(ncall):
            B.mla_indexer_select(q, pooled[i % copies], T, k)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = []
    for _ in range(5):
        e0.record()
        graph.replay()
        e1.record()
        torch.cuda.synchronize()
        per.append(e0.elapsed_time(e1) * 1e3 / ncall)
    sel["call_us"] = sorted(per)[len(per) // 2]
    del graph
    out["calls"].append(sel)
    del keys, pooled
    torch.cuda.empty_cache()
    return out


def _bench_sparse_step(B, dev, reps):
    """The sparse model's verify step for one DSV3-like layer at a 32K cache:
    the indexer's incremental pool update for the L new tokens, the top-512
    window selection (2048 positions per verify row), and the sparse verify
    over those positions, as one CUDA graph of steps over rotating layers;
    events around its replays.  L = 1 and 4."""
    import torch
    from mla_attention_speculative_gb300.inputs import DSV3, make_case
    T, d, kw = 32768, 128, 512
    out = {"geometry": f"DSV3-like H=128 512/128/128, T = {T}; indexer keys bf16 [1, T, {d}], "
                       f"top {kw} windows = {4 * kw} positions", "calls": []}
    g = torch.Generator(device=dev).manual_seed(5200)
    layers = 4
    for L in (1, 4):
        cases = [make_case(DSV3, L, [T], seed=5300 + L * 10 + i, device=dev)
                 for i in range(layers)]
        keys = [torch.randn(1, T, d, generator=g, device=dev).to(torch.bfloat16)
                for _ in range(layers)]
        pooled = [torch.zeros((1, T // 4, d), device=dev) for _ in range(layers)]
        for i in range(layers):
            B.mla_indexer_pool_update(keys[i], T, T, pooled[i], B.IndexerPoolState())
        qi = torch.randn(1, L, d, generator=g, device=dev)
        lens_dev = torch.tensor([T], dtype=torch.int32, device=dev)

        def step(i):
            c = cases[i % layers]
            st = B.IndexerPoolState()
            st.length, st.batch, st.dim = T - L, 1, d   # the pool before this step
            B.mla_indexer_pool_update(keys[i % layers], T, L, pooled[i % layers], st)
            _, pos = B.mla_indexer_select(qi, pooled[i % layers], T, kw)
            B.mla_verify_attention_sparse(c.q_nope, c.q_rope, c.c_kv, c.k_rope, c.W_UK, c.W_UV,
                                          [T], pos, cache_lens_dev=lens_dev)
        for i in range(layers):
            step(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(2 * layers):
                step(i)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        per = []
        for _ in range(max(5, reps)):
            e0.record()
            graph.replay()
            e1.record()
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3 / (2 * layers))
        out["calls"].append({"L": L, "us_per_step": sorted(per)[len(per) // 2],
                             "launches_per_step": 6})
        del graph, cases, keys, pooled
        torch.cuda.empty_cache()
    return out


def _bench_snapshots(B, dev, peaks, reps):
    """The rollback state's convolution snapshots: S (s = 3 state words per
    channel) concatenated with T (n = 5 new activations, channel-fastest) into
    X, and k = 3 snapshot windows of s words written from the row, for
    H = 8192 channels and Q = 1 or 64 sequences.  The fused kernel (one load
    per row) against the ordinary path (the concatenation, then one copy per
    window that reads X back), forced by giving the three windows one
    destination.  Device time per call from a CUDA graph of back-to-back
    calls (launch gaps inside the call included, host time not); four input
    copies rotate so Q = 64 reads from HBM."""
    import torch
    s_, n_, k_, H = 3, 5, 3, 8192
    out = {"geometry": f"s = {s_}, n = {n_}, k = {k_} windows of s, H = {H}, 32-bit words, "
                       "S and X [Q][H][s(+n)], T [Q][n][H]", "calls": []}
    g = torch.Generator(device=dev).manual_seed(5100)
    for Q in (1, 64):
        copies = 4 if Q > 1 else 1
        rows = H * Q
        ss, ts, xs = (1, s_, H * s_), (H, 1, H * n_), (1, s_ + n_, H * (s_ + n_))

        def words(nw):
            return torch.randint(-2**31, 2**31 - 1, (nw,), generator=g, device=dev,
                                 dtype=torch.int32)
        bufs = [dict(S=words(rows * s_), T=words(rows * n_), X=words(rows * (s_ + n_)),
                     C=words(k_ * rows * s_)) for _ in range(copies)]
        fused_w = [(n_ - k_ + 1 + j, j * rows * s_, H * s_) for j in range(k_)]
        same_w = [(n_ - k_ + 1 + j, 0, H * s_) for j in range(k_)]
        ent = {"Q": Q}
        for name, wins in (("fused", fused_w), ("separate", same_w)):
            def call(i, wins=wins):
                b = bufs[i % copies]
                return B.mla_concat_snapshots(b["S"], ss, b["T"], ts, b["X"], xs, s_, n_, H, Q,
                                              b["C"], wins)
            ran_fused = call(0)
            assert ran_fused == (name == "fused")
            n = 4 * copies if Q > 1 else 16
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(n):
                    call(i)
            graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            per = []
            for _ in range(max(5, reps)):
                e0.record()
                graph.replay()
                e1.record()
                torch.cuda.synchronize()
                per.append(e0.elapsed_time(e1) * 1e3 / n)
            us = sorted(per)[len(per) // 2]
            words_moved = rows * ((s_ + n_) * 2 + k_ * s_ * (2 if name == "separate" else 1))
            ent[name] = {"us_per_call": us, "dispatches": 1 if name == "fused" else 1 + k_,
                         "bytes": 4 * words_moved,
                         "hbm_frac": 4 * words_moved / (us * 1e-6) / 1e9 / peaks["hbm_gbs"]}
            del graph
        out["calls"].append(ent)
        del bufs
    torch.cuda.empty_cache()
    return out


def _source_sha(names):
    h = hashlib.sha256()
    for nm in names:
        p = os.path.join(ROOT, "mla_attention_speculative_gb300", "csrc", nm)
        if os.path.exists(p):
            h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {
    "generic_absorbed_attention": ["generic_kernels.cu"],
    "generic_fold": ["generic_kernels.cu"],
    "generic_combine_unembed": ["generic_kernels.cu"],
    "fold_sm103": ["absorbed_sm103.cu", "sm103_ptx.cuh", "mla_api.cu"],
    "absorbed_attn_sm103": ["absorbed_sm103.cu", "sm103_ptx.cuh", "mla_api.cu"],
    "unembed_merge_sm103": ["absorbed_sm103.cu", "sm103_ptx.cuh", "mla_api.cu"],
    "merge_sm103": ["absorbed_sm103.cu", "sm103_ptx.cuh", "mla_api.cu"],
    "unembed_sm103": ["absorbed_sm103.cu", "sm103_ptx.cuh", "mla_api.cu"],
    "expand_sm103": ["materialised_sm103.cu", "sm103_ptx.cuh"],
    "mat_attn_sm103": ["materialised_sm103.cu", "sm103_ptx.cuh"],
}


def _profile_traffic(kernel: str):
    """dram bytes per launch from a committed ncu summary of this kernel, or None
    if there is none or the kernel's source changed since it was taken."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    want_sha = _source_sha(KERNEL_SOURCES.get(kernel, []))
    for fn in sorted(os.listdir(pdir)):
        if not fn.startswith(kernel + "__"):
            continue
        txt = open(os.path.join(pdir, fn)).read()
        sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", txt)
        tb = re.search(r"dram_bytes_per_launch_full_workload:\s*([0-9.eE+]+)", txt)
        if sha and tb and sha.group(1) == want_sha:
            return float(tb.group(1))
    return None


class NvmlClockSampler:
    """SM clock and clock-event reasons of the bench's GPU, read through NVML
    (the driver's libnvidia-ml, found by the GPU's PCI bus id so that a
    remapped CUDA_VISIBLE_DEVICES cannot point it at another GPU) every half
    millisecond from a background thread, so that even a timed region of a
    few milliseconds gets samples taken while it runs.  Reading only."""

    # clock-event reason bits (nvml.h)
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40}

    def __init__(self, dev_index: int):
        import ctypes
        import threading
        self.ctypes, self.threading = ctypes, threading
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        rt = _cudart()
        bus = ctypes.create_string_buffer(32)
        rt.cudaDeviceGetPCIBusId.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.c_int]
        if rt.cudaDeviceGetPCIBusId(bus, 32, dev_index) != 0:
            raise RuntimeError("cudaDeviceGetPCIBusId failed")
        self.handle = ctypes.c_void_p()
        if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.handle)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByPciBusId failed")
        self.nvml = nvml
        self.get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint(0)
        nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx))  # 1 = SM clock
        self.max_mhz = float(mx.value)
        self.samples, self.reasons, self.run = [], 0, False

    def _loop(self):
        ctypes = self.ctypes
        mhz, rs = ctypes.c_uint(0), ctypes.c_ulonglong(0)
        while self.run:
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                self.samples.append(float(mhz.value))
            if self.get_reasons(self.handle, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(0.0005)

    def start(self):
        self.run = True
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.run = False
        self.thread.join()
        if not self.samples:
            return None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(n for n, bit in self.REASONS.items() if self.reasons & bit),
                "samples": len(self.samples), "source": "nvml"}


def clock_sampler(dev_index: int):
    """NVML sampling when the driver library is there, else nvidia-smi."""
    try:
        return NvmlClockSampler(dev_index)
    except Exception:
        return ClockSampler(dev_index)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(sms)}


# ---------------------------------------------------------------------------
# Inputs
# ---------------------------------------------------------------------------

def _layers(dev, num_layers):
    import torch
    from mla_attention_speculative_gb300.inputs import DSV3, make_case
    layers = []
    for i in range(num_layers):
        c = make_case(DSV3, max(WIDTHS), [CACHE_LEN], dtype=torch.bfloat16, seed=1000 + i)
        layers.append(c)
    return layers


def _cpu_oracle_step(case, heads):
    """One step of the workload on the float64 oracle, restricted to `heads`."""
    import oracle
    f = lambda t: t.float().numpy()
    qn, qr = f(case.q_nope), f(case.q_rope)
    ckv, kr, wuk, wuv = f(case.c_kv), f(case.k_rope), f(case.W_UK), f(case.W_UV)
    for L in WIDTHS:
        oracle.absorbed(qn[:, :L], qr[:, :L], ckv, kr, wuk, wuv, [CACHE_LEN], heads=heads)


def cpu_baseline(case, budget_s=12.0, heads_frac=1):
    """Time the oracle as it stands on this host's cores on a bounded sample:
    whole steps (every head) until about budget_s seconds have passed."""
    H = case.geom.H
    heads = list(range(0, H, heads_frac))
    t0 = time.perf_counter()
    reps = 0
    while True:
        _cpu_oracle_step(case, heads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 20:
            break
    calls = reps * len(WIDTHS) * len(heads) / H
    return {"value": calls / el, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} step(s) of 5 calls (L=1,2,4,8,16, T=8192) on {len(heads)} of "
                      f"{H} heads, float64 numpy"
                      + ("" if len(heads) == H else "; value scaled to all heads")
                      + f" ({el:.1f} s)"}


# ---------------------------------------------------------------------------
# Reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    import torch
    from mla_attention_speculative_gb300.inputs import DSV3, make_case
    case = make_case(DSV3, max(WIDTHS), [CACHE_LEN], dtype=torch.bfloat16, seed=1000)
    H = DSV3.H
    # Every head when the run is short enough (about 60 step-equivalents of the
    # whole layer); otherwise an evenly spaced sample, so the run stays within
    # a few minutes.  The oracle has a per-call cost that does not depend on
    # the heads, so a small sample would understate its throughput.
    n_heads = max(8, min(H, H * 60 // max(1, args.steps + args.warmup)))
    heads = list(range(0, H, H // n_heads))[:n_heads]
    for _ in range(args.warmup):
        _cpu_oracle_step(case, heads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _cpu_oracle_step(case, heads)
    el = time.perf_counter() - t0
    calls = args.steps * len(WIDTHS) * len(heads) / H
    value = calls / el
    ms_per_step = el * 1e3 / args.steps * H / len(heads)
    sample = (f"each step = 5 calls (L=1,2,4,8,16, T=8192) on {len(heads)} of {H} heads, "
              "float64 numpy oracle" + ("" if len(heads) == H else "; value scaled to all heads"))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "host CPU"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    from mla_attention_speculative_gb300 import binding as B
    from mla_attention_speculative_gb300 import build_lib
    build_lib.build()
    B.lib()

    peaks = _peaks()
    layers = _layers(dev, NUM_LAYERS)
    geom = layers[0].geom
    g = B.make_geometry(geom.H, geom.r, geom.n, geom.v, geom.rope, torch.bfloat16)

    # device-resident inputs for every layer
    # Each layer's latent cache is one packed [1, T, r + rope] buffer (c_kv and
    # k_rope are views with a row stride of r + rope elements), so the L new
    # rows of a call are one contiguous region.
    D = []
    for c in layers:
        d = {k: getattr(c, k).to(dev) for k in ("q_nope", "q_rope", "W_UK", "W_UV")}
        packed = torch.cat([c.c_kv, c.k_rope], dim=-1).to(dev)
        d["packed"] = packed
        d["c_kv"] = packed[..., :c.geom.r]
        d["k_rope"] = packed[..., c.geom.r:]
        D.append(d)
    lens = [CACHE_LEN]
    lens_dev = torch.tensor(lens, dtype=torch.int32, device=dev)
    ws = {L: B.new_workspace(B.mla_workspace_bytes(g, L, lens, "auto"), dev) for L in WIDTHS}
    outs = {L: torch.empty((1, L, geom.H, geom.v), dtype=torch.bfloat16, device=dev)
            for L in WIDTHS}
    q = [{L: (d["q_nope"][:, :L].contiguous(), d["q_rope"][:, :L].contiguous())
          for L in WIDTHS} for d in D]
    branches = {}

    def call(li, L, stream=None):
        d = D[li]
        qn, qr = q[li][L]
        _, br = B.mla_verify_attention(qn, qr, d["c_kv"], d["k_rope"], d["W_UK"], d["W_UV"],
                                       lens, mode="auto", out=outs[L], workspace=ws[L],
                                       cache_lens_dev=lens_dev, stream=stream)
        branches[L] = br

    # step s uses layers (5*(s%2) + i): two alternating halves of the ten layers
    def step(s):
        base = len(WIDTHS) * (s % 2)
        for i, L in enumerate(WIDTHS):
            call((base + i) % NUM_LAYERS, L)

    # warm-up (eager), then capture one graph per half
    for s in range(max(args.warmup, 3)):
        step(s)
    torch.cuda.synchronize()
    graphs = []
    cap_stream = torch.cuda.Stream(dev)
    for half in range(2):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap_stream):
            step(half)
        graphs.append(gr)
    for s in range(max(args.warmup, 3)):
        graphs[s % 2].replay()
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    # ---- timed region: K graph-replayed steps --------------------------------
    sampler = clock_sampler(local)
    sampler.start()
    if isinstance(sampler, ClockSampler):
        time.sleep(0.3)  # nvidia-smi needs a moment before its first line
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for s in range(args.steps):
        graphs[s % 2].replay()
    e1.record()
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    value = job_rate(args.steps * len(WIDTHS), world, ms / 1e3)
    ms_per_step = ms / args.steps

    # ---- per-kernel device time (events around each launch, eager steps) -----
    B.mla_kernel_timing_read(reset=True)
    B.mla_kernel_timing_enable(True)
    for s in range(args.steps):
        step(s)
    torch.cuda.synchronize()
    B.mla_kernel_timing_enable(False)
    ktimes = B.mla_kernel_timing_read(reset=True)
    launches_per_step = sum(n for n, _ in ktimes.values()) / args.steps
    dominant = max(ktimes, key=lambda k: ktimes[k][1])
    n_dom, ms_dom = ktimes[dominant]
    # algorithmic work of the dominant kernel summed over its launches
    bytes_sum = flops_sum = 0.0
    for L in WIDTHS:
        w = _work(dominant, L, CACHE_LEN)
        if w is None:
            continue
        bytes_sum += w[0] * args.steps
        flops_sum += w[1] * args.steps
    dur_s = ms_dom / 1e3
    t_b = bytes_sum / (peaks["hbm_gbs"] * 1e9)
    t_f = flops_sum / (peaks["bf16_tflops"] * 1e12)
    if t_b >= t_f:
        roof = {"bound": "hbm", "achieved": bytes_sum / dur_s / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops_sum / dur_s / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    tr = _profile_traffic(dominant)
    roof["traffic"] = tr
    roof["kernel"] = dominant
    roof["peak_source"] = f"of {peaks['source']}"
    roof["avg_launch_us"] = ms_dom * 1e3 / max(n_dom, 1)

    # ---- per-width us/call (graph of one call per layer, rotating) -----------
    per_L = {}
    for L in WIDTHS:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=cap_stream):
            for li in range(NUM_LAYERS):
                call(li, L)
        gr.replay()
        torch.cuda.synchronize()
        reps = max(3, args.steps // 5)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            gr.replay()
        b.record()
        torch.cuda.synchronize()
        per_L[str(L)] = a.elapsed_time(b) * 1e3 / (reps * NUM_LAYERS)
        del gr

    # ---- end to end: host inputs -> device -> host result, per step ----------
    e2e = _e2e(args, B, D, q, lens, lens_dev, ws, outs, geom, dev, barrier, world)

    shapes = None
    if not args.no_shapes:
        shapes = _bench_shapes(B, dev, peaks, reps=max(3, min(args.steps, 10)),
                               only=args.shape_groups.split(",") if args.shape_groups else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(layers[0])

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD,
                       "geometry": "H=128 r=512 n=128 v=128 rope=64",
                       "branch": {str(L): B.BRANCH_NAMES[branches[L]] for L in WIDTHS},
                       "l2": f"{NUM_LAYERS} rotating layer buffers "
                             f"({_layer_bytes(geom) * NUM_LAYERS / 1e6:.0f} MB) > L2",
                       "timing": "CUDA graph per step, CUDA events on the replay stream",
                       "parallelism": f"replicas x{world}"},
            "us_per_call": ms_per_step * 1e3 / len(WIDTHS),
            "per_width_us_per_call": per_L,
            "per_width_call_roofline": {
                L: call_roofline(B.BRANCH_NAMES[branches[int(L)]], geom, int(L), [CACHE_LEN],
                                 us, peaks) for L, us in per_L.items()},
            "roofline": roof,
            "kernel_ms_per_step": {k: v[1] / args.steps for k, v in ktimes.items()},
            "shapes": shapes,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": int(round(launches_per_step * args.steps)),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def _layer_bytes(geom):
    return (geom.H * geom.n * geom.r + geom.H * geom.r * geom.v
            + CACHE_LEN * (geom.r + geom.rope)) * 2


def _cudart():
    """The CUDA runtime the process already uses (for plain async copies: a
    cudaMemcpyAsync costs the host about a microsecond, a tensor copy_ call
    several)."""
    import ctypes
    for name in ("libcudart.so.13", "/usr/local/cuda/lib64/libcudart.so.13",
                 "/usr/local/cuda/lib64/libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
        except OSError:
            continue
        rt.cudaMemcpyAsync.restype = ctypes.c_int
        rt.cudaMemcpyAsync.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                       ctypes.c_int, ctypes.c_void_p]
        return rt
    raise RuntimeError("no CUDA runtime library found for the end-to-end copies")


def _e2e(args, B, D, q, lens, lens_dev, ws, outs, geom, dev, barrier, world):
    """Same step through the public call, with each step's new inputs (the
    queries of all widths and the L new latent rows per call) copied from
    pinned host memory and the outputs read back to pinned host memory inside
    the timed region.  The queries of a step travel in one copy (each call gets
    views of the staged buffer), each call's new rows in one copy into its
    layer's packed cache, all before the step's first call (so the calls'
    kernels follow one another with no copy between them), and the outputs in
    one copy back.  The copies are plain cudaMemcpyAsync calls on the current
    stream.  The calls are the library's prepared form of the public call
    (binding.PreparedVerifyAttention: the same C entry point, its arguments
    marshalled once for these fixed buffers), as a serving loop would use."""
    import torch
    H, n, v, rope, r = geom.H, geom.n, geom.v, geom.rope, geom.r
    qn_el = {L: L * H * n for L in WIDTHS}
    qr_el = {L: L * H * rope for L in WIDTHS}
    q_total = sum(qn_el[L] + qr_el[L] for L in WIDTHS)
    host_q = torch.empty(q_total, dtype=torch.bfloat16).pin_memory()
    dev_q = torch.empty(q_total, dtype=torch.bfloat16, device=dev)
    views, off = {}, 0
    for L in WIDTHS:
        qn = dev_q[off:off + qn_el[L]].view(1, L, H, n)
        host_q[off:off + qn_el[L]].copy_(q[0][L][0].reshape(-1).cpu())
        off += qn_el[L]
        qr = dev_q[off:off + qr_el[L]].view(1, L, H, rope)
        host_q[off:off + qr_el[L]].copy_(q[0][L][1].reshape(-1).cpu())
        off += qr_el[L]
        views[L] = (qn, qr)
    host_new = {L: D[0]["packed"][:, CACHE_LEN - L:].cpu().pin_memory() for L in WIDTHS}
    out_el = {L: L * H * v for L in WIDTHS}
    dev_out = torch.empty(sum(out_el.values()), dtype=torch.bfloat16, device=dev)
    host_out = torch.empty(dev_out.numel(), dtype=torch.bfloat16).pin_memory()
    ovs, off = {}, 0
    for L in WIDTHS:
        ovs[L] = dev_out[off:off + out_el[L]].view(1, L, H, v)
        off += out_el[L]
    h2d = host_q.numel() * 2 + sum(t.numel() * 2 for t in host_new.values())
    d2h = host_out.numel() * 2
    rt = _cudart()
    stream = torch.cuda.current_stream(dev).cuda_stream
    H2D, D2H = 1, 2
    # (destination, source, bytes) of every input copy of a step, per half of the layers
    ins = []
    for half in range(2):
        cp = [(dev_q.data_ptr(), host_q.data_ptr(), host_q.numel() * 2)]
        for i, L in enumerate(WIDTHS):
            dst = D[(len(WIDTHS) * half + i) % len(D)]["packed"][:, CACHE_LEN - L:]
            assert dst.is_contiguous()
            cp.append((dst.data_ptr(), host_new[L].data_ptr(), host_new[L].numel() * 2))
        ins.append(cp)
    outcp = (host_out.data_ptr(), dev_out.data_ptr(), host_out.numel() * 2)

    def copy(dst, src, nbytes, kind):
        if rt.cudaMemcpyAsync(dst, src, nbytes, kind, stream) != 0:
            raise RuntimeError("cudaMemcpyAsync failed")

    calls = []
    for half in range(2):
        row = []
        for i, L in enumerate(WIDTHS):
            d = D[(len(WIDTHS) * half + i) % len(D)]
            row.append(B.PreparedVerifyAttention(views[L][0], views[L][1], d["c_kv"], d["k_rope"],
                                                 d["W_UK"], d["W_UV"], lens, mode="auto",
                                                 out=ovs[L], workspace=ws[L],
                                                 cache_lens_dev=lens_dev))
        calls.append(row)

    def step(s):
        for dst, src, nbytes in ins[s % 2]:
            copy(dst, src, nbytes, H2D)
        for call in calls[s % 2]:
            call.run()
        copy(*outcp, D2H)
        torch.cuda.current_stream().synchronize()

    for s in range(3):
        step(s)
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s)
    el = time.perf_counter() - t0
    barrier()
    if world > 1:
        import torch.distributed as dist
        el = max_over_ranks(el, dist, dev)
    return {"value": job_rate(args.steps * len(WIDTHS), world, el), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def main():
    global WIDTHS, WORKLOAD
    args = _args()
    if args.widths:
        WIDTHS = tuple(int(x) for x in args.widths.split(","))
        WORKLOAD = WORKLOAD.replace("L=1,2,4,8,16", "L=" + ",".join(map(str, WIDTHS)))
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
