"""Thin Python binding of ``libkvmm.so`` (the C ABI declared in ``include/kvmm.h``).

Argument marshalling only: every function checks the tensors it is given
(device, dtype, contiguity, element count), turns them into raw device
pointers and calls the C entry point of the same name on the current (or
given) CUDA stream.  All computation happens in the library's kernels; there
is no fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

OK, INVALID_ARG, UNSUPPORTED_SHAPE, WORKSPACE_TOO_SMALL, CUDA_ERROR = range(5)
ERR_NULL_BLOCK, ERR_OUT_OF_RANGE, ERR_TIMEOUT = 1, 2, 4
EARLY_READS = DECODE_EARLY_READS = 1
NULL_BLOCK = -1

EXPORTS = ("kv_minmax_update", "page_score_topk", "sparse_paged_decode_attn", "topk_promotion_diff",
           "kvmm_workspace_size", "kvmm_auto_splits", "kvmm_decode_layer_cluster", "kvmm_decode_layer_units",
           "kvmm_status_string",
           "kvmm_last_cuda_error", "page_score_topk_static_scratch", "page_score_topk_attn", "decode_layer", "topk_history_record",
           "topk_stability_rco", "promote_pages", "block_table_update", "kv_meankey_update",
           "page_score_topk_mean", "kv_centroid_build", "page_score_topk_centroid")


class KvmmError(RuntimeError):
    def __init__(self, fn: str, status: int):
        msg = f"{fn}: {status_string(status)} (status {status})"
        if status == CUDA_ERROR:
            msg += f": {load().kvmm_last_cuda_error().decode()}"
        super().__init__(msg)
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("L", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32),
                ("D", ctypes.c_int32), ("T", ctypes.c_int32), ("Pmax", ctypes.c_int32), ("Kmax", ctypes.c_int32),
                ("n_phys", ctypes.c_int64)]

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def __repr__(self) -> str:
        return ("Shape(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")")


def make_shape(B, L, Hq, Hkv, D, T, Pmax, Kmax, n_phys) -> Shape:
    return Shape(B, L, Hq, Hkv, D, T, Pmax, Kmax, n_phys)


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load ``libkvmm.so`` (built by ``paged_kv_cache_minmax_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"kvmm CUDA library not found at {path}: build it first "
                           "(python -m paged_kv_cache_minmax_gb300.build)")
    lib = ctypes.CDLL(path)
    P, I32, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    SP = ctypes.POINTER(Shape)
    lib.kv_minmax_update.argtypes = [SP, I32, P, P, I32, P, P, P, P, P, P, P, P]
    U32 = ctypes.c_uint32
    lib.page_score_topk.argtypes = [SP, I32, P, P, P, P, I32, I32, P, P, P, P, SZ, U32, P, P]
    lib.sparse_paged_decode_attn.argtypes = [SP, I32, P, P, P, P, P, P, P, F32, I32, P, P, P, SZ, U32, P, P]
    lib.topk_promotion_diff.argtypes = [SP, I32, P, P, P, P, P, I32, P, P, P, P, P, P, P]
    lib.page_score_topk_static_scratch.argtypes = [SP, I32, P, P, P, P, I32, I32, P, P, P, P, P]
    lib.page_score_topk_attn.argtypes = [SP, I32, P, P, P, P, P, P, P, I32, I32, F32, P, P, P, P, P, P, SZ, P, P]
    lib.decode_layer.argtypes = [SP, I32, P, P, P, I32, P, P, P, P, P, P, P, P, I32, I32, F32, P, P, P, P, P, P, SZ,
                                 ctypes.c_uint32, P, P]
    lib.topk_history_record.argtypes = [SP, I32, P, P, P, I32, I32, P, P, P, P, P]
    lib.topk_stability_rco.argtypes = [SP, P, P, P, I32, I32, I32, I32, F32, P, P, P, P, P]
    lib.promote_pages.argtypes = [SP, I32, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, P, P]
    lib.block_table_update.argtypes = [SP, P, P, I32, P, P, P]
    lib.kv_meankey_update.argtypes = [SP, I32, P, P, P, P, P, P, P]
    lib.page_score_topk_mean.argtypes = [SP, I32, P, P, P, P, I32, I32, P, P, P, P, SZ, P, P]
    lib.kv_centroid_build.argtypes = [SP, I32, P, P, I32, I32, P, P, P, P, P, P]
    lib.page_score_topk_centroid.argtypes = [SP, I32, P, P, P, I32, P, P, P, P, I32, I32, I32, P, P, P, P, P, P]
    for f in ("kv_minmax_update", "page_score_topk", "sparse_paged_decode_attn", "topk_promotion_diff",
              "page_score_topk_static_scratch", "page_score_topk_attn", "decode_layer", "topk_history_record",
              "topk_stability_rco", "promote_pages", "block_table_update", "kv_meankey_update",
              "page_score_topk_mean", "kv_centroid_build", "page_score_topk_centroid"):
        getattr(lib, f).restype = ctypes.c_int
    lib.kvmm_workspace_size.argtypes = [SP, I32]
    lib.kvmm_workspace_size.restype = SZ
    lib.kvmm_auto_splits.argtypes = [SP]
    lib.kvmm_auto_splits.restype = I32
    lib.kvmm_decode_layer_cluster.argtypes = [SP]
    lib.kvmm_decode_layer_cluster.restype = I32
    lib.kvmm_decode_layer_units.argtypes = [SP]
    lib.kvmm_decode_layer_units.restype = I32
    lib.kvmm_status_string.argtypes = [ctypes.c_int]
    lib.kvmm_status_string.restype = ctypes.c_char_p
    lib.kvmm_last_cuda_error.argtypes = []
    lib.kvmm_last_cuda_error.restype = ctypes.c_char_p
    if path == library_path():
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().kvmm_status_string(status).decode()


def _check(fn: str, status: int) -> None:
    if status != OK:
        raise KvmmError(fn, status)


def _dev(t: torch.Tensor | None, name: str, dtype: torch.dtype, numel: int | None = None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def _stream(stream) -> int | None:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# --------------------------------------------------------------------------- #
def workspace_size(shape: Shape, num_splits: int = 0) -> int:
    return int(load().kvmm_workspace_size(ctypes.byref(shape), num_splits))


def auto_splits(shape: Shape) -> int:
    return int(load().kvmm_auto_splits(ctypes.byref(shape)))


def decode_layer_cluster(shape: Shape) -> int:
    return int(load().kvmm_decode_layer_cluster(ctypes.byref(shape)))


def decode_layer_units(shape: Shape) -> int:
    return int(load().kvmm_decode_layer_units(ctypes.byref(shape)))


def alloc_workspace(shape: Shape, num_splits: int = 0, device="cuda") -> torch.Tensor:
    """A zero-filled workspace (uint8) of ``workspace_size`` bytes, rounded to 16."""
    n = workspace_size(shape, num_splits)
    if n == 0:
        raise KvmmError("kvmm_workspace_size", UNSUPPORTED_SHAPE)
    return torch.zeros((n + 15) // 16 * 16, dtype=torch.uint8, device=device)


def kv_minmax_update(shape: Shape, layer: int, new_k, new_v, n_new: int, tok_begin, tok_end, k_pool, v_pool,
                     block_table, meta, err=None, stream=None) -> None:
    s = shape
    if (new_k is None) != (new_v is None):
        raise ValueError("new_k and new_v are given together or not at all")
    rows = s.B * s.Hkv * n_new * s.D
    args = (ctypes.byref(s), layer,
            _dev(new_k, "new_k", torch.bfloat16, rows, optional=True),
            _dev(new_v, "new_v", torch.bfloat16, rows, optional=True), n_new,
            _dev(tok_begin, "tok_begin", torch.int32, s.B), _dev(tok_end, "tok_end", torch.int32, s.B),
            _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(v_pool, "v_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(block_table, "block_table", torch.int32, s.B * s.L * s.Hkv * s.Pmax),
            _dev(meta, "meta", torch.bfloat16, s.B * s.L * s.Hkv * s.Pmax * 2 * s.D),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("kv_minmax_update", load().kv_minmax_update(*args))


def page_score_topk(shape: Shape, layer: int, q, meta, seq_len, rescore_mask, K: int, sel_idx, sel_cnt,
                    workspace, err=None, scores_out=None, group_reduce: int = 0, stream=None,
                    early_reads: bool = False) -> None:
    """Score and select for one layer.  ``early_reads``: no kernel still running when this launch starts
    writes seq_len, the layer's rescore_mask row or its metadata rows (``KVMM_EARLY_READS``)."""
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(meta, "meta", torch.bfloat16, units * s.Pmax * 2 * s.D),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), K, group_reduce,
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(), EARLY_READS if early_reads else 0,
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("page_score_topk", load().page_score_topk(*args))


def page_score_topk_static_scratch(shape: Shape, layer: int, q, meta, seq_len, rescore_mask, K: int, sel_idx,
                                   sel_cnt, err=None, scores_out=None, group_reduce: int = 0, stream=None) -> None:
    """page_score_topk with the library's fixed device scratch instead of a caller workspace.

    For callers that cannot allocate device memory at call time; the scratch
    is shared by every call on a device, so calls must not overlap on the GPU.
    """
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(meta, "meta", torch.bfloat16, units * s.Pmax * 2 * s.D),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), K, group_reduce,
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("page_score_topk_static_scratch", load().page_score_topk_static_scratch(*args))


def sparse_paged_decode_attn(shape: Shape, layer: int, q, k_pool, v_pool, block_table, seq_len, sel_idx, sel_cnt,
                             out, workspace, lse=None, err=None, sm_scale: float = 0.0, num_splits: int = 0,
                             stream=None, early_reads: bool = False) -> None:
    """Attention over the kept selections of one layer.  ``early_reads`` (automatic split count only): no
    kernel still running when this launch starts writes seq_len or the layer's block-table rows."""
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(v_pool, "v_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(block_table, "block_table", torch.int32, units * s.Pmax),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            float(sm_scale), num_splits, _dev(out, "out", torch.float32, s.B * s.Hq * s.D),
            _dev(lse, "lse", torch.float32, s.B * s.Hq, optional=True),
            _dev(workspace, "workspace", torch.uint8, optional=True),
            0 if workspace is None else workspace.numel(), EARLY_READS if early_reads else 0,
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("sparse_paged_decode_attn", load().sparse_paged_decode_attn(*args))


def page_score_topk_attn(shape: Shape, layer: int, q, meta, k_pool, v_pool, block_table, seq_len, rescore_mask,
                         K: int, sel_idx, sel_cnt, out, workspace, lse=None, err=None, scores_out=None,
                         group_reduce: int = 0, sm_scale: float = 0.0, stream=None) -> None:
    """page_score_topk then sparse_paged_decode_attn on the new selection, in one launch."""
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(meta, "meta", torch.bfloat16, units * s.Pmax * 2 * s.D),
            _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(v_pool, "v_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(block_table, "block_table", torch.int32, units * s.Pmax),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), K, group_reduce,
            float(sm_scale),
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(out, "out", torch.float32, s.B * s.Hq * s.D),
            _dev(lse, "lse", torch.float32, s.B * s.Hq, optional=True),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("page_score_topk_attn", load().page_score_topk_attn(*args))


def decode_layer(shape: Shape, layer: int, q, new_k, new_v, n_new: int, tok_begin, tok_end, k_pool, v_pool,
                 block_table, meta, seq_len, rescore_mask, K: int, sel_idx, sel_cnt, out, lse=None, err=None,
                 scores_out=None, group_reduce: int = 0, sm_scale: float = 0.0, workspace=None,
                 stream=None, early_reads: bool = False) -> None:
    """Append (optional), score, select and attend for one layer in one launch.  ``early_reads``: no kernel
    still running when this launch starts (after a kvmm call: that call alone) writes anything this call reads
    of seq_len, tok_begin, tok_end, rescore_mask, block_table and meta (``KVMM_DECODE_EARLY_READS``); two
    calls for the same layer back to back do not meet this."""
    s = shape
    units = s.B * s.L * s.Hkv
    if (new_k is None) != (new_v is None):
        raise ValueError("new_k and new_v are given together or not at all")
    app = new_k is not None
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(new_k, "new_k", torch.bfloat16, s.B * s.Hkv * max(n_new, 1) * s.D, optional=True),
            _dev(new_v, "new_v", torch.bfloat16, s.B * s.Hkv * max(n_new, 1) * s.D, optional=True),
            int(n_new) if app else 0,
            _dev(tok_begin, "tok_begin", torch.int32, s.B, optional=not app),
            _dev(tok_end, "tok_end", torch.int32, s.B, optional=not app),
            _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(v_pool, "v_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(block_table, "block_table", torch.int32, units * s.Pmax),
            _dev(meta, "meta", torch.bfloat16, units * s.Pmax * 2 * s.D),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), K, group_reduce,
            float(sm_scale),
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(out, "out", torch.float32, s.B * s.Hq * s.D),
            _dev(lse, "lse", torch.float32, s.B * s.Hq, optional=True),
            _dev(workspace, "workspace", torch.uint8, optional=True), 0 if workspace is None else workspace.numel(),
            DECODE_EARLY_READS if early_reads else 0,
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("decode_layer", load().decode_layer(*args))


def topk_promotion_diff(shape: Shape, layer: int, rescore_mask, prev_idx, prev_cnt, cur_idx, cur_cnt, promoted,
                        promoted_cnt, evicted=None, evicted_cnt=None, total_promoted=None, commit: bool = True,
                        err=None, stream=None) -> None:
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer,
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True),
            _dev(prev_idx, "prev_idx", torch.int32, units * s.Kmax), _dev(prev_cnt, "prev_cnt", torch.int32, units),
            _dev(cur_idx, "cur_idx", torch.int32, units * s.Kmax), _dev(cur_cnt, "cur_cnt", torch.int32, units),
            int(bool(commit)), _dev(promoted, "promoted", torch.int32, units * s.Kmax),
            _dev(promoted_cnt, "promoted_cnt", torch.int32, units),
            _dev(evicted, "evicted", torch.int32, units * s.Kmax, optional=True),
            _dev(evicted_cnt, "evicted_cnt", torch.int32, units, optional=True),
            _dev(total_promoted, "total_promoted", torch.int32, 1, optional=True),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("topk_promotion_diff", load().topk_promotion_diff(*args))


def topk_history_record(shape: Shape, layer: int, sel_idx, sel_cnt, seq_len, slot: int, hist_idx, hist_cnt,
                        hist_pages, err=None, stream=None) -> None:
    """Store ``layer``'s selections in ring slot ``slot`` (hist_idx [W,B,L,Hkv,Kmax], hist_cnt [W,B,L,Hkv],
    hist_pages [W,B], all int32; W is taken from hist_pages)."""
    s = shape
    units = s.B * s.L * s.Hkv
    W = hist_pages.shape[0]
    args = (ctypes.byref(s), layer, _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax),
            _dev(sel_cnt, "sel_cnt", torch.int32, units), _dev(seq_len, "seq_len", torch.int32, s.B), W, slot,
            _dev(hist_idx, "hist_idx", torch.int32, W * units * s.Kmax),
            _dev(hist_cnt, "hist_cnt", torch.int32, W * units), _dev(hist_pages, "hist_pages", torch.int32, W * s.B),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("topk_history_record", load().topk_history_record(*args))


def topk_stability_rco(shape: Shape, hist_idx, hist_cnt, hist_pages, n: int, head: int, lag: int, rco_unit,
                       stability=None, unstable=None, unstable_frac: float = 0.25, err=None, stream=None) -> None:
    """Per-unit mean RCO of selections ``lag`` steps apart over the last ``n`` recorded steps (newest in slot
    ``head``), the per-head stability and the unstable mask; see kvmm.h."""
    s = shape
    units = s.B * s.L * s.Hkv
    W = hist_pages.shape[0]
    args = (ctypes.byref(s), _dev(hist_idx, "hist_idx", torch.int32, W * units * s.Kmax),
            _dev(hist_cnt, "hist_cnt", torch.int32, W * units), _dev(hist_pages, "hist_pages", torch.int32, W * s.B),
            W, n, head, lag, float(unstable_frac), _dev(rco_unit, "rco_unit", torch.float32, units),
            _dev(stability, "stability", torch.float32, s.L * s.Hkv, optional=True),
            _dev(unstable, "unstable", torch.uint8, s.L * s.Hkv, optional=True),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("topk_stability_rco", load().topk_stability_rco(*args))


def _host(t: torch.Tensor, name: str, numel: int):
    """A host-side bf16 store (pinned, or pageable where the device reads pageable memory)."""
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous bfloat16")
    if t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def promote_pages(shape: Shape, layer: int, rescore_mask, promoted, promoted_cnt, evicted, evicted_cnt, host_k,
                  host_v, k_pool, v_pool, block_table, moved=None, freed=None, freed_cnt=None, max_ctas: int = 0,
                  err=None, stream=None) -> None:
    """Promoted pages from the host store (host_k [B,L,Hkv,Pmax,T,D], host_v [B,L,Hkv,Pmax,D,T], bf16) into the
    blocks of evicted pages, and the table rewrite; see kvmm.h."""
    s = shape
    units = s.B * s.L * s.Hkv
    page = s.T * s.D
    args = (ctypes.byref(s), layer, _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True),
            _dev(promoted, "promoted", torch.int32, units * s.Kmax),
            _dev(promoted_cnt, "promoted_cnt", torch.int32, units),
            _dev(evicted, "evicted", torch.int32, units * s.Kmax), _dev(evicted_cnt, "evicted_cnt", torch.int32, units),
            _host(host_k, "host_k", units * s.Pmax * page), _host(host_v, "host_v", units * s.Pmax * page),
            _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * page), _dev(v_pool, "v_pool", torch.bfloat16, s.n_phys * page),
            _dev(block_table, "block_table", torch.int32, units * s.Pmax),
            _dev(moved, "moved", torch.int32, units, optional=True),
            _dev(freed, "freed", torch.int32, units * s.Kmax, optional=True),
            _dev(freed_cnt, "freed_cnt", torch.int32, units, optional=True), int(max_ctas),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("promote_pages", load().promote_pages(*args))


def block_table_update(shape: Shape, idx, val, block_table, err=None, stream=None) -> None:
    """block_table.view(-1)[idx[i]] = val[i]; idx (int64) and val (int32) on the device or in pinned host memory."""
    s = shape
    n = int(idx.numel())
    if int(val.numel()) != n:
        raise ValueError("idx and val differ in length")
    for t, name, dt in ((idx, "idx", torch.int64), (val, "val", torch.int32)):
        if t.dtype != dt or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous {dt}")
    args = (ctypes.byref(s), idx.data_ptr() if n else None, val.data_ptr() if n else None, n,
            _dev(block_table, "block_table", torch.int32, s.B * s.L * s.Hkv * s.Pmax),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("block_table_update", load().block_table_update(*args))


def kv_meankey_update(shape: Shape, layer: int, tok_begin, tok_end, k_pool, block_table, mean, err=None,
                      stream=None) -> None:
    """Mean key of every page meeting [tok_begin, tok_end) (tok_begin None = 0) into mean [B,L,Hkv,Pmax,D]."""
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(tok_begin, "tok_begin", torch.int32, s.B, optional=True),
            _dev(tok_end, "tok_end", torch.int32, s.B), _dev(k_pool, "k_pool", torch.bfloat16, s.n_phys * s.T * s.D),
            _dev(block_table, "block_table", torch.int32, units * s.Pmax),
            _dev(mean, "mean", torch.bfloat16, units * s.Pmax * s.D), _dev(err, "err", torch.int32, 1, optional=True),
            _stream(stream))
    _check("kv_meankey_update", load().kv_meankey_update(*args))


def page_score_topk_mean(shape: Shape, layer: int, q, mean, seq_len, rescore_mask, K: int, sel_idx, sel_cnt,
                         workspace, err=None, scores_out=None, group_reduce: int = 0, stream=None) -> None:
    """page_score_topk with the mean key (mean [B,L,Hkv,Pmax,D]) as the page's row."""
    s = shape
    units = s.B * s.L * s.Hkv
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(mean, "mean", torch.bfloat16, units * s.Pmax * s.D),
            _dev(seq_len, "seq_len", torch.int32, s.B),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), K, group_reduce,
            _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax), _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(workspace, "workspace", torch.uint8), workspace.numel(),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("page_score_topk_mean", load().page_score_topk_mean(*args))


def centroid_rows(shape: Shape, R: int) -> int:
    """Cmax = ceil(Pmax / R): the centroid rows a unit holds at most."""
    return (shape.Pmax + R - 1) // R


def kv_centroid_build(shape: Shape, layer: int, mean, seq_len, R: int, n_iter: int, cent, assign, member_off, members,
                      err=None, stream=None) -> None:
    """KVDrive's centroid level over the layer's pages' mean keys: spatial blocks of R pages, then n_iter Lloyd
    iterations.  cent [B,L,Hkv,Cmax,D] bf16, assign [B,L,Hkv,Pmax], member_off [B,L,Hkv,Cmax+1],
    members [B,L,Hkv,Pmax] int32 (Cmax = ceil(Pmax / R))."""
    s = shape
    units = s.B * s.L * s.Hkv
    cmax = centroid_rows(s, R)
    args = (ctypes.byref(s), layer, _dev(mean, "mean", torch.bfloat16, units * s.Pmax * s.D),
            _dev(seq_len, "seq_len", torch.int32, s.B), int(R), int(n_iter),
            _dev(cent, "cent", torch.bfloat16, units * cmax * s.D), _dev(assign, "assign", torch.int32, units * s.Pmax),
            _dev(member_off, "member_off", torch.int32, units * (cmax + 1)),
            _dev(members, "members", torch.int32, units * s.Pmax), _dev(err, "err", torch.int32, 1, optional=True),
            _stream(stream))
    _check("kv_centroid_build", load().kv_centroid_build(*args))


def page_score_topk_centroid(shape: Shape, layer: int, q, mean, seq_len, R: int, cent, member_off, members,
                             rescore_mask, M: int, K: int, sel_idx, sel_cnt, err=None, centroid_scores_out=None,
                             scores_out=None, group_reduce: int = 0, stream=None) -> None:
    """The two-level selection: score the centroids, expand the M best, keep the K best of their pages."""
    s = shape
    units = s.B * s.L * s.Hkv
    cmax = centroid_rows(s, R)
    args = (ctypes.byref(s), layer, _dev(q, "q", torch.bfloat16, s.B * s.Hq * s.D),
            _dev(mean, "mean", torch.bfloat16, units * s.Pmax * s.D), _dev(seq_len, "seq_len", torch.int32, s.B),
            int(R), _dev(cent, "cent", torch.bfloat16, units * cmax * s.D),
            _dev(member_off, "member_off", torch.int32, units * (cmax + 1)),
            _dev(members, "members", torch.int32, units * s.Pmax),
            _dev(rescore_mask, "rescore_mask", torch.uint8, s.L * s.Hkv, optional=True), int(M), int(K),
            int(group_reduce), _dev(sel_idx, "sel_idx", torch.int32, units * s.Kmax),
            _dev(sel_cnt, "sel_cnt", torch.int32, units),
            _dev(centroid_scores_out, "centroid_scores_out", torch.float32, s.B * s.Hkv * cmax, optional=True),
            _dev(scores_out, "scores_out", torch.float32, s.B * s.Hkv * s.Pmax, optional=True),
            _dev(err, "err", torch.int32, 1, optional=True), _stream(stream))
    _check("page_score_topk_centroid", load().page_score_topk_centroid(*args))
