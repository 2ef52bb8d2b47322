"""CPU oracle for MinMax page selection and sparse paged GQA decode attention.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use this package; the product path never imports it, and it
imports nothing from the product package.  The arithmetic lives in
``kvmm_oracle.c`` (plain C, double precision, one unit at a time, written from
the FlexiCache page's "Core method" sections 2 and 3 and its "head-level block
table" paragraph, and from KVDrive's description of Quest scoring).  This
module only builds that file with gcc and marshals numpy arrays into it.

bf16 tensors are passed as ``numpy.uint16`` arrays of their raw bit patterns.

Parity pins for every function are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvmm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

ERR_NULL_BLOCK = 1
ERR_OUT_OF_RANGE = 2

_lock = threading.Lock()
_lib = None
_prebuilt = False  # set on variants loaded from an already-built library


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the C source (gcc, -O2, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not _prebuilt:
            build()
        lib = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_unit_append.argtypes = [P, P, I64, I32, I32, P, I32, I32, P, P]
        lib.oracle_unit_append.restype = I32
        lib.oracle_unit_minmax.argtypes = [P, I64, I32, I32, P, I32, I32, I32, P]
        lib.oracle_unit_minmax.restype = I32
        lib.oracle_unit_scores.argtypes = [P, I32, I32, P, I32, I32, P]
        lib.oracle_unit_scores.restype = None
        lib.oracle_topk.argtypes = [P, I32, I32, P]
        lib.oracle_topk.restype = I32
        lib.oracle_set_difference.argtypes = [P, I32, P, I32, P]
        lib.oracle_set_difference.restype = I32
        lib.oracle_unit_sparse_attention.argtypes = [P, I32, I32, I32, P, P, I64, P, I32, P, I32, D, P, P]
        lib.oracle_unit_sparse_attention.restype = I32
        lib.oracle_unit_dense_attention.argtypes = [P, I32, I32, I32, P, P, I64, P, I32, D, P, P]
        lib.oracle_unit_dense_attention.restype = I32
        lib.oracle_unit_promote.argtypes = [P, I32, I64, P, I32, P, I32, P, P, P, P, I32, I32, P, P]
        lib.oracle_unit_promote.restype = I32
        lib.oracle_table_update.argtypes = [P, I64, I64, P, P, I64]
        lib.oracle_table_update.restype = I32
        lib.oracle_unit_meankey.argtypes = [P, I64, I32, I32, P, I32, I32, I32, P]
        lib.oracle_unit_meankey.restype = I32
        lib.oracle_unit_mean_scores.argtypes = [P, I32, I32, P, I32, I32, P]
        lib.oracle_unit_mean_scores.restype = None
        lib.oracle_unit_page_mass.argtypes = [P, I32, I32, I32, P, I64, P, I32, D, P]
        lib.oracle_unit_page_mass.restype = I32
        lib.oracle_centroid_build.argtypes = [P, I32, I32, I32, I32, P, P, P, P]
        lib.oracle_centroid_build.restype = I32
        lib.oracle_centroid_select.argtypes = [P, I32, I32, P, I32, P, I32, P, P, I32, I32, I32, P, P, P, P, P, P]
        lib.oracle_centroid_select.restype = I32
        lib.oracle_rco.argtypes = [P, I32, P, I32, I32]
        lib.oracle_rco.restype = D
        lib.oracle_unit_stability.argtypes = [P, P, P, I32, I32, I32]
        lib.oracle_unit_stability.restype = D
        lib.oracle_classify.argtypes = [P, I32, D, P]
        lib.oracle_classify.restype = None
        lib.oracle_unit_step.argtypes = [P, P, I64, I32, I32, P, I32, P, P, P, P, I32, I32, I32, I32,
                                         P, P, P, P, P, P, P, D, P, P]
        lib.oracle_unit_step.restype = I32
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, f"bf16 bit patterns expected as uint16, got {a.dtype}"
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


# --------------------------------------------------------------------------- #
# per-unit functions                                                          #
# --------------------------------------------------------------------------- #
def unit_append(k_pool, v_pool, T, bt_row, tok_begin, tok_end, new_k, new_v) -> int:
    """Write token rows [tok_begin, tok_end) into the pools (in place); returns error bits."""
    D = k_pool.shape[-1]
    n_phys = k_pool.size // (T * D)
    return int(_load().oracle_unit_append(_ptr(k_pool), _ptr(v_pool), n_phys, T, D, _ptr(_i32(bt_row)),
                                          tok_begin, tok_end, _ptr(_u16(new_k)), _ptr(_u16(new_v))))


def unit_minmax(k_pool, T, bt_row, seq_len, page_begin=0, page_end=None, meta=None):
    """MinMax metadata ``[P][2][D]`` (uint16 bf16 bits) of one unit; returns (meta, err)."""
    k_pool = _u16(k_pool)
    D = k_pool.shape[-1]
    n_phys = k_pool.size // (T * D)
    bt_row = _i32(bt_row)
    P = (seq_len + T - 1) // T
    if page_end is None:
        page_end = P
    if meta is None:
        meta = np.zeros((max(len(bt_row), P), 2, D), dtype=np.uint16)
    err = _load().oracle_unit_minmax(_ptr(k_pool), n_phys, T, D, _ptr(bt_row), seq_len, page_begin,
                                     page_end, _ptr(meta))
    return meta, int(err)


def unit_scores(q, meta, P, group_reduce=0) -> np.ndarray:
    """Scores ``[P]`` (float64) of one unit; q is ``[G][D]`` bf16 bits."""
    q = _u16(q)
    meta = _u16(meta)
    G, D = q.shape
    out = np.zeros(P, dtype=np.float64)
    _load().oracle_unit_scores(_ptr(q), G, D, _ptr(meta), P, group_reduce, _ptr(out))
    return out


def topk(scores, K) -> np.ndarray:
    """Top-K page indices (ascending) of a score vector; ties to the lower index."""
    scores = np.ascontiguousarray(scores, dtype=np.float64)
    sel = np.zeros(max(K, 1), dtype=np.int32)
    n = _load().oracle_topk(_ptr(scores), len(scores), K, _ptr(sel))
    assert n >= 0
    return sel[:n].copy()


def set_difference(a, b) -> np.ndarray:
    """a \\ b for two ascending integer lists."""
    a, b = _i32(a), _i32(b)
    out = np.zeros(max(len(a), 1), dtype=np.int32)
    n = _load().oracle_set_difference(_ptr(a), len(a), _ptr(b), len(b), _ptr(out))
    return out[:n].copy()


def unit_promote(bt_row, n_phys, promoted, evicted, host_k, host_v, k_pool, v_pool, T):
    """Promotion of one unit in place: bt_row (int32 [Pmax]) and the pools (uint16 bf16 bits [n_phys, T*D]) are
    updated from the unit's host pages (uint16 [Pmax, T*D]).  Returns (err, moved, freed)."""
    bt = np.ascontiguousarray(bt_row, dtype=np.int32)
    assert bt_row.flags["C_CONTIGUOUS"] and bt_row.dtype == np.int32 and bt.ctypes.data == bt_row.ctypes.data
    pr, ev = _i32(promoted), _i32(evicted)
    D = host_k.shape[-1] // T
    freed = np.zeros(max(len(ev), 1), dtype=np.int32)
    moved = np.zeros(1, dtype=np.int32)
    err = _load().oracle_unit_promote(_ptr(bt), len(bt), int(n_phys), _ptr(pr), len(pr), _ptr(ev), len(ev),
                                      _ptr(_u16(host_k)), _ptr(_u16(host_v)), _ptr(k_pool), _ptr(v_pool), T, D,
                                      _ptr(freed), _ptr(moved))
    m = min(len(pr), len(ev))
    return int(err), int(moved[0]), freed[:max(0, len(ev) - m)].copy()


def table_update(table, n_phys, idx, val) -> int:
    """table (int32, C-contiguous, updated in place).flat[idx[i]] = val[i] in order; returns the error bits."""
    assert table.dtype == np.int32 and table.flags["C_CONTIGUOUS"]
    idx = np.ascontiguousarray(idx, dtype=np.int64)
    val = _i32(val)
    return int(_load().oracle_table_update(_ptr(table), table.size, int(n_phys), _ptr(idx), _ptr(val), len(idx)))


def unit_meankey(k_pool, T, bt_row, seq_len, page_begin=0, page_end=None, mean=None):
    """Mean keys (uint16 bf16 bits [Pmax, D]) of pages [page_begin, page_end); returns (mean, err)."""
    k_pool = _u16(k_pool)
    bt = _i32(bt_row)
    D = k_pool.shape[-1]
    n_phys = k_pool.size // (T * D)
    P = len(bt)
    if mean is None:
        mean = np.zeros((P, D), dtype=np.uint16)
    err = _load().oracle_unit_meankey(_ptr(k_pool), n_phys, T, D, _ptr(bt), int(seq_len), int(page_begin),
                                      P if page_end is None else int(page_end), _ptr(mean))
    return mean, int(err)


def unit_mean_scores(q, mean, P, group_reduce=0) -> np.ndarray:
    q, mean = _u16(q), _u16(mean)
    G, D = q.shape
    out = np.zeros(max(P, 1), dtype=np.float64)
    _load().oracle_unit_mean_scores(_ptr(q), G, D, _ptr(mean), int(P), int(group_reduce), _ptr(out))
    return out[:P].copy()


def centroid_build(mean, R, n_iter):
    """KVDrive's centroid level over a unit's pages' mean keys ``mean`` (uint16 bf16 bits [P, D]): Lloyd's
    k-means from spatial blocks of R pages, n_iter iterations.  Returns (cent [n_c, D] uint16, assign [P],
    off [n_c + 1], members [P]) -- the pages of centroid j are members[off[j]:off[j+1]], ascending."""
    mean = _u16(mean)
    P, D = mean.shape
    n_c = (P + R - 1) // R
    cent = np.zeros((max(n_c, 1), D), dtype=np.uint16)
    assign = np.zeros(max(P, 1), dtype=np.int32)
    off = np.zeros(n_c + 1, dtype=np.int32)
    members = np.zeros(max(P, 1), dtype=np.int32)
    got = _load().oracle_centroid_build(_ptr(mean), P, D, int(R), int(n_iter), _ptr(cent), _ptr(assign), _ptr(off),
                                        _ptr(members))
    assert got == n_c
    return cent[:n_c].copy(), assign[:P].copy(), off, members[:P].copy()


def centroid_select(q, mean, cent, off, members, M, K, group_reduce=0):
    """The two-level search of one unit: score the centroids, expand the M best, keep the K best of their
    pages.  Returns a dict: cs (centroid scores), chosen (centroids, ascending), cand (their pages, ascending),
    ps (the candidates' scores), sel (the selection, ascending)."""
    q, mean, cent = _u16(q), _u16(mean), _u16(cent)
    off, members = _i32(off), _i32(members)
    G, D = q.shape
    P = mean.shape[0]
    n_c = len(off) - 1
    cs = np.zeros(max(n_c, 1), dtype=np.float64)
    chosen = np.zeros(max(n_c, 1), dtype=np.int32)
    cand = np.zeros(max(P, 1), dtype=np.int32)
    ps = np.zeros(max(P, 1), dtype=np.float64)
    sel = np.zeros(max(P, 1), dtype=np.int32)
    n_cand = ctypes.c_int32(0)
    cnt = _load().oracle_centroid_select(_ptr(q), G, D, _ptr(mean), P, _ptr(cent), n_c, _ptr(off), _ptr(members),
                                         int(M), int(K), int(group_reduce), _ptr(cs), _ptr(chosen), _ptr(cand),
                                         ctypes.addressof(n_cand), _ptr(ps), _ptr(sel))
    n = n_cand.value
    return {"cs": cs[:n_c].copy(), "chosen": chosen[:min(M, n_c)].copy(), "cand": cand[:n].copy(),
            "ps": ps[:n].copy(), "sel": sel[:cnt].copy()}


def unit_page_mass(q, k_pool, T, bt_row, seq_len, scale=0.0) -> np.ndarray:
    """Dense attention mass [G, P] of every page (softmax over every token below seq_len)."""
    q, k_pool, bt = _u16(q), _u16(k_pool), _i32(bt_row)
    G, D = q.shape
    n_phys = k_pool.size // (T * D)
    P = (int(seq_len) + T - 1) // T
    out = np.zeros((G, max(P, 1)), dtype=np.float64)
    _load().oracle_unit_page_mass(_ptr(q), G, D, T, _ptr(k_pool), n_phys, _ptr(bt), int(seq_len), float(scale),
                                  _ptr(out))
    return out[:, :P].copy()


def rco(a, b, P) -> float:
    """Random-Corrected Overlap of page sets a and b drawn from P pages (FlexiCache, "Core insight")."""
    a, b = _i32(a), _i32(b)
    return float(_load().oracle_rco(_ptr(a), len(a), _ptr(b), len(b), int(P)))


def unit_stability(idx, cnt, pages, lag) -> float:
    """Mean RCO of steps ``lag`` apart over a window given newest first: idx [n, kmax], cnt [n], pages [n]."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    cnt, pages = _i32(cnt), _i32(pages)
    n, kmax = idx.shape
    return float(_load().oracle_unit_stability(_ptr(idx), _ptr(cnt), _ptr(pages), kmax, n, int(lag)))


def classify(stability, frac) -> np.ndarray:
    """1 for the round(frac * n) entries of lowest stability (ties: lower index first)."""
    st = np.ascontiguousarray(stability, dtype=np.float64).ravel()
    out = np.zeros(max(st.size, 1), dtype=np.uint8)
    _load().oracle_classify(_ptr(st), st.size, float(frac), _ptr(out))
    return out[:st.size].copy()


def unit_sparse_attention(q, k_pool, v_pool, T, bt_row, seq_len, sel, scale=0.0):
    """Attention of q ``[G][D]`` over the selected pages; returns (out [G][D], lse [G], err)."""
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    G, D = q.shape
    n_phys = k_pool.size // (T * D)
    sel = _i32(sel)
    out = np.zeros((G, D), dtype=np.float64)
    lse = np.zeros(G, dtype=np.float64)
    err = _load().oracle_unit_sparse_attention(_ptr(q), G, D, T, _ptr(k_pool), _ptr(v_pool), n_phys,
                                               _ptr(_i32(bt_row)), seq_len, _ptr(sel), len(sel),
                                               float(scale), _ptr(out), _ptr(lse))
    return out, lse, int(err)


def unit_dense_attention(q, k_pool, v_pool, T, bt_row, seq_len, scale=0.0):
    """Attention of q over every token < seq_len; returns (out, lse, err)."""
    q, k_pool, v_pool = _u16(q), _u16(k_pool), _u16(v_pool)
    G, D = q.shape
    n_phys = k_pool.size // (T * D)
    out = np.zeros((G, D), dtype=np.float64)
    lse = np.zeros(G, dtype=np.float64)
    err = _load().oracle_unit_dense_attention(_ptr(q), G, D, T, _ptr(k_pool), _ptr(v_pool), n_phys,
                                              _ptr(_i32(bt_row)), seq_len, float(scale), _ptr(out),
                                              _ptr(lse))
    return out, lse, int(err)


class UnitState:
    """Mutable per-unit state for :func:`unit_step`: pools, metadata and selection."""

    def __init__(self, k_pool, v_pool, T, bt_row, meta, K):
        self.k_pool = _u16(k_pool)
        self.v_pool = _u16(v_pool)
        self.T = T
        self.bt_row = _i32(bt_row)
        self.meta = _u16(meta)
        self.K = K
        self.sel = np.zeros(max(K, 1), dtype=np.int32)
        self.sel_cnt = np.zeros(1, dtype=np.int32)
        self.promoted = np.zeros(max(K, 1), dtype=np.int32)
        self.evicted = np.zeros(max(K, 1), dtype=np.int32)
        self.n_promoted = np.zeros(1, dtype=np.int32)
        self.n_evicted = np.zeros(1, dtype=np.int32)
        self.scores = np.zeros(max(len(self.bt_row), 1), dtype=np.float64)


def unit_step(st: UnitState, seq_len, new_k, new_v, q, rescore, group_reduce=0, scale=0.0):
    """One decode step of one unit in the method's order (see ``oracle_unit_step``).

    Returns (out [G][D], lse [G], err); ``st`` carries the selection and the
    promoted / evicted lists of this step.
    """
    q = _u16(q)
    G, D = q.shape
    n_phys = st.k_pool.size // (st.T * D)
    out = np.zeros((G, D), dtype=np.float64)
    lse = np.zeros(G, dtype=np.float64)
    nk = None if new_k is None else _u16(new_k)
    nv = None if new_v is None else _u16(new_v)
    err = _load().oracle_unit_step(
        _ptr(st.k_pool), _ptr(st.v_pool), n_phys, st.T, D, _ptr(st.bt_row), seq_len, _ptr(nk), _ptr(nv),
        _ptr(st.meta), _ptr(q), G, int(bool(rescore)), st.K, group_reduce, _ptr(st.sel), _ptr(st.sel_cnt),
        _ptr(st.promoted), _ptr(st.n_promoted), _ptr(st.evicted), _ptr(st.n_evicted), _ptr(st.scores),
        float(scale), _ptr(out), _ptr(lse))
    return out, lse, int(err)


def load_variant(so_path: str):
    """A separate instance of this module bound to another build of the oracle.

    Used by the mutation tests, which compile deliberately broken copies of
    ``kvmm_oracle.c`` and check that the pins reject them.
    """
    import importlib.util

    spec = importlib.util.spec_from_file_location(f"_oracle_variant_{abs(hash(so_path))}", __file__)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._LIB_PATH = so_path
    mod._prebuilt = True
    return mod


def rescored(unstable: bool, step: int, period: int = 16) -> bool:
    """Rerank schedule: an unstable head rescores every step, a stable head when step % period == 0.

    FlexiCache page, "Core method, 3. Periodic reranking and incremental
    promotion" (stable heads rerank every 16 steps by default).
    """
    return bool(unstable) or step % period == 0
