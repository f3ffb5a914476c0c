"""Thin ctypes binding of libmla.so (argument marshalling only).

Every function here has the C entry point's name and forwards to it.  The
tensors are PyTorch CUDA tensors: PyTorch provides device memory and the
current stream, nothing else.  Every step of the attention runs in the
library's kernels; if the library is missing this module raises instead of
falling back to anything.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_CUDA = -4
MLA_ERR_TIMEOUT = -5

MODES = {"auto": 0, "absorbed": 1, "materialised": 2}
BRANCH_ABSORBED = 1
BRANCH_MATERIALISED = 2
BRANCH_NAMES = {1: "absorbed", 2: "materialised"}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}


class MlaError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({detail})")


class Geometry(ctypes.Structure):
    _fields_ = [("num_heads", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32),
                ("qk_nope_dim", ctypes.c_int32), ("v_dim", ctypes.c_int32),
                ("rope_dim", ctypes.c_int32), ("softmax_scale", ctypes.c_float),
                ("dtype", ctypes.c_int32)]


_lib = None

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIGS = {
    "mla_max_absorbed_queries": (_I64, [_I32, _I32, _I32, _I64]),
    "mla_max_absorbed_queries_batch": (_I64, [_I32, _I32, _I32, _P, _I32]),
    "mla_select_branch": (_I32, [_P, _I32, _P, _I32, _I32, _P]),
    "mla_workspace_bytes": (_I32, [_P, _I32, _I32, _P, _I32, _P]),
    "mla_verify_attention": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P,
                                    _I32, _I32, _P, _I32, _I32, _I32, _I32, _P, _P,
                                    ctypes.c_size_t, _P, _P]),
    "mla_verify_attention_noalloc": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P,
                                            _P, _P, _I32, _I32, _P, _I32, _I32, _I32, _P,
                                            _P, _P]),
    "mla_check_page_table": (_I32, [_P, _I32, _I32, _P, _I32, _I32]),
    "mla_sparse_workspace_bytes": (_I32, [_P, _I32, _I32, _P, _I32, _P]),
    "mla_indexer_pool_update": (_I32, [_P, _I32, _I64, _I64, _I32, _I32, _I64, _I32, _I32, _P,
                                       _I64, _P, _P, _P]),
    "mla_indexer_select_workspace_bytes": (_I32, [_I32, _I32, _I64, _P]),
    "mla_indexer_select": (_I32, [_P, _P, _I64, _I32, _I32, _I64, _I32, _I32, _P, _P, _P,
                                  ctypes.c_size_t, _P]),
    "mla_verify_attention_sparse": (_I32, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _P, _P, _P,
                                           _I32, _I32, _P, _I32, _P, _I32, _I32, _I32, _P, _P,
                                           ctypes.c_size_t, _P]),
    "mla_select_draft_cap": (_I32, [ctypes.c_double, _P, _I32, _P, _I32, _I32, _P]),
    "mla_concat_snapshots": (_I32, [_P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _I64, _P,
                                    _I32, _P, _P]),
    "mla_rollback_valid_prefix": (_I32, [_P, _I32, _I32, _P, _P, _I32, _I32, _I32, _I32, _I32,
                                         _P, _P]),
    "mla_kernel_timing_enable": (_I32, [_I32]),
    "mla_kernel_timing_read": (_I32, [ctypes.c_char_p, ctypes.c_size_t, _P, _P, _I32, _P,
                                      _I32]),
    "mla_device_status": (_I32, [_P, _I32]),
    "mla_selftest_bounded_wait": (_I32, [_P]),
    "mla_status_string": (ctypes.c_char_p, [_I32]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_version": (_I32, []),
}


def lib() -> ctypes.CDLL:
    """Load libmla.so (built in-tree by build_lib); raise if it is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run "
                               "`python -m mla_attention_speculative_gb300.build_lib`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def mla_last_error() -> str:
    return lib().mla_last_error().decode()


def _check(status: int, where: str):
    if status != MLA_OK:
        raise MlaError(status, where, mla_last_error())


def _lens_array(cache_lens: Sequence[int]):
    arr = (ctypes.c_int32 * len(cache_lens))(*[int(t) for t in cache_lens])
    return arr


def make_geometry(H, r, n, v, rope, dtype=torch.bfloat16, scale: Optional[float] = None):
    return Geometry(int(H), int(r), int(n), int(v), int(rope),
                    float(scale) if scale is not None else 0.0, DTYPES[dtype])


_GEOMS = {}


def _geometry(H, r, n, v, rope, dtype, scale):
    """A Geometry per distinct shape, built once (the call only reads it)."""
    key = (H, r, n, v, rope, dtype, scale)
    g = _GEOMS.get(key)
    if g is None:
        g = _GEOMS[key] = make_geometry(H, r, n, v, rope, dtype, scale)
    return g


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _current_stream(dev: torch.device) -> int:
    """The raw handle of the current CUDA stream of `dev` (PyTorch's fast accessor
    when present, else the public one)."""
    if _raw_stream is not None:
        return _raw_stream(dev.index if dev.index is not None else torch.cuda.current_device())
    return torch.cuda.current_stream(dev).cuda_stream


def mla_max_absorbed_queries(r: int, n: int, v: int, cache_len: int = 0) -> int:
    return int(lib().mla_max_absorbed_queries(r, n, v, cache_len))


def mla_max_absorbed_queries_batch(r: int, n: int, v: int, cache_lens: Sequence[int]) -> int:
    arr = _lens_array(cache_lens)
    return int(lib().mla_max_absorbed_queries_batch(r, n, v, arr, len(cache_lens)))


def mla_select_branch(geom: Geometry, L: int, cache_lens: Sequence[int], mode="auto") -> int:
    arr = _lens_array(cache_lens)
    out = ctypes.c_int32(0)
    _check(lib().mla_select_branch(ctypes.byref(geom), L, arr, len(cache_lens),
                                   MODES.get(mode, mode), ctypes.byref(out)),
           "mla_select_branch")
    return out.value


def mla_workspace_bytes(geom: Geometry, L: int, cache_lens: Sequence[int], mode="auto") -> int:
    arr = _lens_array(cache_lens)
    out = ctypes.c_size_t(0)
    _check(lib().mla_workspace_bytes(ctypes.byref(geom), len(cache_lens), L, arr,
                                     MODES.get(mode, mode), ctypes.byref(out)),
           "mla_workspace_bytes")
    return out.value


def mla_sparse_workspace_bytes(geom: Geometry, L: int, cache_lens: Sequence[int],
                               topk_len: int) -> int:
    arr = _lens_array(cache_lens)
    out = ctypes.c_size_t(0)
    _check(lib().mla_sparse_workspace_bytes(ctypes.byref(geom), len(cache_lens), L, arr,
                                            int(topk_len), ctypes.byref(out)),
           "mla_sparse_workspace_bytes")
    return out.value


def mla_check_page_table(page_table, cache_lens: Sequence[int], page_size: int,
                         num_pages: int) -> None:
    """Host-side range check of a page table (any int array-like [B, max_pages]);
    raises MlaError (MLA_ERR_INVALID_ARG) naming the first bad entry."""
    t = torch.as_tensor(page_table, dtype=torch.int32).cpu().contiguous()
    if t.dim() != 2:
        raise ValueError("page_table must be [batch, max_pages]")
    lens = _lens_array(cache_lens)
    _check(lib().mla_check_page_table(t.data_ptr(), t.shape[0], t.shape[1], lens, int(page_size),
                                      int(num_pages)), "mla_check_page_table")


def mla_select_draft_cap(p: float, verify_cost: Sequence[float], drafter_cost,
                         max_cap: int):
    """(best cap, [speedup(0), ..., speedup(limit)]) from a measured verify-cost
    curve (verify_cost[w-1] = cost of a pass over w rows) and the drafter's
    cost (one number, or one per cap)."""
    dr = [float(drafter_cost)] if isinstance(drafter_cost, (int, float)) else \
        [float(x) for x in drafter_cost]
    vc = (ctypes.c_double * len(verify_cost))(*[float(x) for x in verify_cost])
    dc = (ctypes.c_double * len(dr))(*dr)
    n_out = max(1, min(int(max_cap), len(verify_cost) - 1) + 1)
    sp = (ctypes.c_double * n_out)()
    cap = lib().mla_select_draft_cap(float(p), vc, len(verify_cost), dc, len(dr), int(max_cap), sp)
    if cap < 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_select_draft_cap", mla_last_error())
    limit = min(int(max_cap), len(verify_cost) - 1, len(dr) - 1 if len(dr) > 1 else 1 << 30)
    return int(cap), [sp[i] for i in range(limit + 1)]


def new_workspace(nbytes: int, device) -> torch.Tensor:
    """An (uninitialised) workspace of at least `nbytes` bytes."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


class SnapshotWindow(ctypes.Structure):
    _fields_ = [("window_start", ctypes.c_int32), ("cache_offset", ctypes.c_int64),
                ("sequence_stride", ctypes.c_int64)]


def _words(t: torch.Tensor) -> torch.Tensor:
    """A 32-bit tensor seen as uint32 words (no copy)."""
    if t.element_size() != 4:
        raise ValueError("snapshot buffers hold 32-bit words")
    return t


def mla_concat_snapshots(S, s_strides, T, t_strides, X, x_strides, s: int, n: int, H: int,
                         Q: int, cache, windows, stream=None) -> bool:
    """Concatenate S || T into X and write the snapshot windows into `cache`
    (flat 32-bit device tensors; strides in words).  windows: list of
    (window_start, cache_offset, sequence_stride).  Returns True when the
    fused single-load kernel ran, False for the ordinary path."""
    for t in (S, T, X, cache):
        _words(t)
    arr = (SnapshotWindow * max(1, len(windows)))(*[SnapshotWindow(*w) for w in windows])
    st = lambda v: (ctypes.c_int64 * 3)(*[int(x) for x in v])
    if stream is None:
        stream = _current_stream(X.device)
    fused = ctypes.c_int32(0)
    _check(lib().mla_concat_snapshots(_ptr(S), st(s_strides), _ptr(T), st(t_strides), _ptr(X),
                                      st(x_strides), s, n, H, Q, _ptr(cache), cache.numel(),
                                      arr, len(windows), stream, ctypes.byref(fused)),
           "mla_concat_snapshots")
    return bool(fused.value)


def mla_rollback_valid_prefix(blocks, r: int, cell_pos, cell_seq, p0: int, p1: int = -1,
                              seq: int = 0, n_streams: int = 1, stream=None) -> torch.Tensor:
    """Leading valid pooled blocks after a rollback from p0 (device int32
    tensor of one element).  blocks: int32 [n_blocks, 8 + r]; cell_pos: int32
    [n_cells]; cell_seq: int64 [n_cells] owner bit masks."""
    dev = cell_pos.device
    out = torch.empty(1, dtype=torch.int32, device=dev)
    _dense(blocks=blocks, cell_pos=cell_pos, cell_seq=cell_seq)
    if stream is None:
        stream = _current_stream(dev)
    _check(lib().mla_rollback_valid_prefix(_ptr(blocks), blocks.shape[0], r, _ptr(cell_pos),
                                           _ptr(cell_seq), cell_pos.numel(), p0, p1, seq,
                                           n_streams, _ptr(out), stream),
           "mla_rollback_valid_prefix")
    return out


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _dense(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (row-major)")


def mla_device_status(clear: bool = True) -> int:
    """Wait for the device, then raise MlaError if a kernel's bounded wait ran out."""
    code = ctypes.c_int32(0)
    _check(lib().mla_device_status(ctypes.byref(code), 1 if clear else 0), "mla_device_status")
    return code.value


def mla_selftest_bounded_wait(stream=None) -> None:
    """Launch the library's failure-path self-test (a bounded wait that runs out
    after about a second); mla_device_status then raises MLA_ERR_TIMEOUT."""
    if stream is None:
        stream = _current_stream(torch.device("cuda", torch.cuda.current_device()))
    _check(lib().mla_selftest_bounded_wait(stream), "mla_selftest_bounded_wait")


def cache_strides(c_kv: torch.Tensor, k_rope: torch.Tensor, paged: bool):
    """(c_kv row stride, k_rope row stride, rows between sequences) in elements."""
    if c_kv.stride(-1) != 1 or k_rope.stride(-1) != 1:
        raise ValueError("cache rows must be contiguous in their last dimension")
    cs, ks = c_kv.stride(1), k_rope.stride(1)
    if paged:
        if c_kv.stride(0) != c_kv.shape[1] * cs or k_rope.stride(0) != k_rope.shape[1] * ks:
            raise ValueError("paged cache pages must be contiguous runs of rows")
        return cs, ks, 0
    if c_kv.stride(0) % cs or k_rope.stride(0) % ks or \
            c_kv.stride(0) // cs != k_rope.stride(0) // ks:
        raise ValueError("c_kv and k_rope must have the same rows per sequence")
    return cs, ks, c_kv.stride(0) // cs


def _verify_args(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, mode, out, workspace,
                 page_table, cache_lens_dev, scale, noalloc=False):
    """Checks, defaults and the C arguments of mla_verify_attention up to (not
    including) the stream and the branch pointer.  Returns (args, out, dev,
    keep), keep holding every tensor the arguments point into.  With
    ``noalloc`` the arguments are those of mla_verify_attention_noalloc (no
    mode, no workspace)."""
    B, L, H, n = q_nope.shape
    rope = q_rope.shape[-1]
    r = W_UK.shape[-1]
    v = W_UV.shape[-1]
    dev = q_nope.device
    _dense(q_nope=q_nope, q_rope=q_rope, W_UK=W_UK, W_UV=W_UV, out=out, page_table=page_table)
    geom = _geometry(H, r, n, v, rope, q_nope.dtype, scale)
    lens = [int(t) for t in cache_lens]
    arr = _lens_array(lens)
    paged = page_table is not None
    cs, ks, seq = cache_strides(c_kv, k_rope, paged)
    if cache_lens_dev is None:
        cache_lens_dev = torch.tensor(lens, dtype=torch.int32, device=dev)
    if out is None:
        out = torch.empty((B, L, H, v), dtype=q_nope.dtype, device=dev)
    page_size = c_kv.shape[1] if paged else 0
    max_pages = page_table.shape[1] if paged else 0
    num_pages = c_kv.shape[0] if paged else 0
    args = [ctypes.byref(geom), _ptr(q_nope), _ptr(q_rope), _ptr(c_kv), _ptr(k_rope), cs, ks, seq,
            _ptr(W_UK), _ptr(W_UV), _ptr(cache_lens_dev), arr, B, L, _ptr(page_table), page_size,
            max_pages, num_pages]
    if noalloc:
        args += [_ptr(out)]
    else:
        m = MODES.get(mode, mode)
        if workspace is None:  # (a given workspace that is too small is rejected by the call)
            workspace = new_workspace(mla_workspace_bytes(geom, L, lens, m), dev)
        args += [m, _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size()]
    keep = (q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, page_table, cache_lens_dev, out, workspace)
    return args, out, dev, keep


def mla_verify_attention(q_nope: torch.Tensor, q_rope: torch.Tensor, c_kv: torch.Tensor,
                         k_rope: torch.Tensor, W_UK: torch.Tensor, W_UV: torch.Tensor,
                         cache_lens: Sequence[int], mode="auto",
                         out: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         page_table: Optional[torch.Tensor] = None,
                         cache_lens_dev: Optional[torch.Tensor] = None,
                         scale: Optional[float] = None, stream=None):
    """One verify call through the C ABI.  Returns (out, branch).

    q_nope [B,L,H,n], q_rope [B,L,H,rope], W_UK [H,n,r], W_UV [H,r,v]; the
    cache is c_kv [B,Tmax,r] / k_rope [B,Tmax,rope] (contiguous) or
    [num_pages,page,r] / [num_pages,page,rope] with ``page_table`` [B,max_pages].
    ``out`` and ``workspace`` are allocated with torch when not given.
    """
    args, out, dev, _ = _verify_args(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, mode,
                                     out, workspace, page_table, cache_lens_dev, scale)
    if stream is None:
        stream = _current_stream(dev)
    branch = ctypes.c_int32(0)
    st = lib().mla_verify_attention(*args, stream, ctypes.byref(branch))
    _check(st, "mla_verify_attention")
    return out, branch.value


class PreparedVerifyAttention:
    """mla_verify_attention with its arguments marshalled once.

    For a caller that repeats a call on the same device buffers, as a serving
    loop does when it writes each step's queries and new cache rows into fixed
    tensors: the tensors, shapes, cache lengths and mode are fixed when the
    object is made (with the same checks and defaults as
    mla_verify_attention); ``run()`` issues the call on the current stream
    (or ``stream``) with whatever the buffers hold then, and returns the
    branch taken.  The tensors must outlive the object.  The library entry
    point and its results are the same as for mla_verify_attention.
    """

    def __init__(self, q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, mode="auto",
                 out=None, workspace=None, page_table=None, cache_lens_dev=None, scale=None):
        args, self.out, dev, self._keep = _verify_args(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV,
                                                       cache_lens, mode, out, workspace,
                                                       page_table, cache_lens_dev, scale)
        self._fn = lib().mla_verify_attention
        types = _SIGS["mla_verify_attention"][1]
        # plain ints become ctypes values now, so a run converts nothing
        self._args = [types[i](a) if isinstance(a, int) else a for i, a in enumerate(args)]
        self._dev = dev.index if dev.index is not None else torch.cuda.current_device()
        self._branch = ctypes.c_int32(0)
        self._branch_ref = ctypes.byref(self._branch)

    def run(self, stream=None) -> int:
        if stream is None:
            stream = (_raw_stream(self._dev) if _raw_stream is not None else
                      torch.cuda.current_stream(self._dev).cuda_stream)
        st = self._fn(*self._args, stream, self._branch_ref)
        if st != MLA_OK:
            _check(st, "mla_verify_attention")
        return self._branch.value


def mla_kernel_timing_enable(on: bool = True) -> None:
    """Bracket every library kernel launch with CUDA events (benchmark instrumentation)."""
    _check(lib().mla_kernel_timing_enable(1 if on else 0), "mla_kernel_timing_enable")


def mla_kernel_timing_read(reset: bool = True) -> dict:
    """{kernel name: (launches, total device ms)} of the kernels launched since
    the last reset (waits for their events)."""
    cap = 64
    names = ctypes.create_string_buffer(4096)
    launches = (ctypes.c_int32 * cap)()
    ms = (ctypes.c_double * cap)()
    n = ctypes.c_int32(0)
    _check(lib().mla_kernel_timing_read(names, 4096, launches, ms, cap, ctypes.byref(n),
                                        1 if reset else 0), "mla_kernel_timing_read")
    keys = names.value.decode().split(";") if n.value else []
    return {k: (int(launches[i]), float(ms[i])) for i, k in enumerate(keys[:cap])
            if launches[i] > 0}


def mla_verify_attention_noalloc(q_nope: torch.Tensor, q_rope: torch.Tensor,
                                 c_kv: torch.Tensor, k_rope: torch.Tensor,
                                 W_UK: torch.Tensor, W_UV: torch.Tensor,
                                 cache_lens: Sequence[int], out: Optional[torch.Tensor] = None,
                                 page_table: Optional[torch.Tensor] = None,
                                 cache_lens_dev: Optional[torch.Tensor] = None,
                                 scale: Optional[float] = None, stream=None):
    """Absorbed-branch verify call that uses the library's static scratch
    instead of a workspace (for callers that cannot allocate device memory).
    Same tensors and checks as :func:`mla_verify_attention`; returns (out, branch)."""
    args, out, dev, _ = _verify_args(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens,
                                     None, out, None, page_table, cache_lens_dev, scale,
                                     noalloc=True)
    if stream is None:
        stream = _current_stream(dev)
    branch = ctypes.c_int32(0)
    st = lib().mla_verify_attention_noalloc(*args, stream, ctypes.byref(branch))
    _check(st, "mla_verify_attention_noalloc")
    return out, branch.value


def mla_verify_attention_sparse(q_nope: torch.Tensor, q_rope: torch.Tensor, c_kv: torch.Tensor,
                                k_rope: torch.Tensor, W_UK: torch.Tensor, W_UV: torch.Tensor,
                                cache_lens: Sequence[int], topk: torch.Tensor,
                                out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None,
                                page_table: Optional[torch.Tensor] = None,
                                cache_lens_dev: Optional[torch.Tensor] = None,
                                scale: Optional[float] = None, stream=None) -> torch.Tensor:
    """Absorbed verify call over selected cached positions (the sparse model's
    top-k attention).  ``topk`` is an int32 device tensor [B, L, k]: verify row
    l of sequence b attends to the positions topk[b, l, :] that lie in
    [0, T_b - L + l] (others, e.g. -1 padding, are skipped).  The other
    tensors are those of :func:`mla_verify_attention`.  Returns out."""
    _dense(topk=topk)
    if topk.dtype != torch.int32 or topk.dim() != 3 or tuple(topk.shape[:2]) != \
            tuple(q_nope.shape[:2]):
        raise ValueError("topk must be int32 [B, L, k] matching q_nope's B and L")
    k = topk.shape[2]
    args, out, dev, _ = _verify_args(q_nope, q_rope, c_kv, k_rope, W_UK, W_UV, cache_lens, None,
                                     out, None, page_table, cache_lens_dev, scale, noalloc=True)
    geom_ref, L, arr = args[0], args[13], args[11]
    if workspace is None:
        nbytes = ctypes.c_size_t(0)
        _check(lib().mla_sparse_workspace_bytes(geom_ref, len(cache_lens), L, arr, int(k),
                                                ctypes.byref(nbytes)),
               "mla_sparse_workspace_bytes")
        workspace = new_workspace(nbytes.value, dev)
    if stream is None:
        stream = _current_stream(dev)
    # (geometry .. B, L) + (topk, k) + (page table .. num_pages) + (out, workspace, bytes)
    cargs = args[:14] + [_ptr(topk), int(k)] + args[14:18] + \
        [_ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), stream]
    _check(lib().mla_verify_attention_sparse(*cargs), "mla_verify_attention_sparse")
    return out


class IndexerPoolState(ctypes.Structure):
    """What a pool of indexer keys describes (mla_indexer_pool_state_t)."""
    _fields_ = [("length", ctypes.c_int64), ("batch", ctypes.c_int32), ("dim", ctypes.c_int32)]

    def __init__(self):
        super().__init__(-1, 0, 0)


def mla_indexer_pool_update(keys: torch.Tensor, cache_len: int, new_tokens: int,
                            pooled: torch.Tensor, state: IndexerPoolState, padded: bool = False,
                            stream=None) -> bool:
    """Pool the indexer keys of one step.  keys [batch, Tmax, dim] (bf16 or
    fp32, rows contiguous), pooled fp32 [batch, cap, dim]; ``state`` is
    updated.  Returns True when the incremental (tail-only) path ran."""
    if keys.dim() != 3 or keys.stride(-1) != 1 or not pooled.is_contiguous() or \
            pooled.dtype != torch.float32:
        raise ValueError("keys must be [batch, T, dim] with contiguous rows, pooled fp32 "
                         "[batch, cap, dim] contiguous")
    Bn, _, d = keys.shape
    inc = ctypes.c_int32(0)
    if stream is None:
        stream = _current_stream(keys.device)
    _check(lib().mla_indexer_pool_update(
        _ptr(keys), DTYPES[keys.dtype], keys.stride(1), keys.stride(0) // keys.stride(1), Bn, d,
        int(cache_len), int(new_tokens), 1 if padded else 0, _ptr(pooled), pooled.shape[1],
        ctypes.byref(state), ctypes.byref(inc), stream), "mla_indexer_pool_update")
    return bool(inc.value)


def mla_indexer_select(q: torch.Tensor, pooled: torch.Tensor, cache_len: int, k_windows: int,
                       stream=None):
    """(windows [batch, S, k], positions [batch, S, 4k]) int32: each new
    token's k best visible windows, ascending, and their positions."""
    _dense(q=q, pooled=pooled)
    Bn, S, d = q.shape
    dev = q.device
    wins = torch.empty((Bn, S, k_windows), dtype=torch.int32, device=dev)
    pos = torch.empty((Bn, S, 4 * k_windows), dtype=torch.int32, device=dev)
    nbytes = ctypes.c_size_t(0)
    _check(lib().mla_indexer_select_workspace_bytes(Bn, S, int(cache_len), ctypes.byref(nbytes)),
           "mla_indexer_select_workspace_bytes")
    ws = new_workspace(nbytes.value, dev)
    if stream is None:
        stream = _current_stream(dev)
    _check(lib().mla_indexer_select(_ptr(q), _ptr(pooled), pooled.shape[1], Bn, d, int(cache_len),
                                    S, int(k_windows), _ptr(wins), _ptr(pos), _ptr(ws),
                                    ws.numel(), stream), "mla_indexer_select")
    return wins, pos
