"""Shared helpers for the GPU parity tests: pull one unit's bytes to the host,
run the oracle on them and compare with what the CUDA path produced.

Tolerances (fixed by the target, written here once):
  * MinMax metadata: bit-exact.
  * page scores: |s_gpu - s_oracle| <= 1e-5 * max |s_oracle| of the unit
    (fp32 versus double accumulation).
  * selection: the GPU selection equals the exact top-K of its own fp32
    scores (bit-exact, lowest-index ties); against the oracle's selection a
    page may differ only if its oracle score lies within 1e-5 * |s_K| of the
    oracle's K-th score s_K (a counted tie).
  * attention: max |out_gpu - out_oracle| <= 2e-3 and
    sum |out_gpu - out_oracle| / sum |out_oracle| <= 1e-3 (mean relative),
    with the oracle run over the GPU's selection; same bounds on lse.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
from paged_kv_cache_minmax_gb300.workloads import bf16_bits

SCORE_RTOL = 1e-5
TIE_RTOL = 1e-5
OUT_MAX_ABS = 2e-3
OUT_MEAN_REL = 1e-3


@dataclass
class Stats:
    units: int = 0
    ties: int = 0
    abs_err_sum: float = 0.0
    ref_abs_sum: float = 0.0
    max_abs: float = 0.0
    lse_max_abs: float = 0.0
    notes: list = field(default_factory=list)

    @property
    def mean_rel(self) -> float:
        return self.abs_err_sum / max(self.ref_abs_sum, 1e-30)

    def check(self):
        assert self.max_abs <= OUT_MAX_ABS, f"max-abs {self.max_abs:.3e} > {OUT_MAX_ABS}"
        assert self.mean_rel <= OUT_MEAN_REL, f"mean-rel {self.mean_rel:.3e} > {OUT_MEAN_REL}"
        assert self.lse_max_abs <= OUT_MAX_ABS, f"lse max-abs {self.lse_max_abs:.3e}"


def unit_pool(wl, b, l, h, full=None):
    """Host pools and block-table row for one unit.

    With ``full`` = (k_host, v_host) the whole pool is used with the real
    table row (the indirection itself is under test); otherwise the unit's
    resident pages are gathered into a compact pool and the row is remapped.
    """
    cfg = wl.cfg
    row = wl.block_table[b, l, h].cpu().numpy().astype(np.int32)
    if full is not None:
        return full[0], full[1], row
    seq = int(wl.seq_len[b])
    P = -(-seq // cfg.T)
    valid = np.nonzero((row[:P] >= 0) & (row[:P] < wl.n_phys))[0]
    idx = torch.as_tensor(row[valid], dtype=torch.long, device=wl.k_pool.device)
    kp = bf16_bits(wl.k_pool.index_select(0, idx)) if len(valid) else np.zeros((0, cfg.T, cfg.D), np.uint16)
    vp = bf16_bits(wl.v_pool.index_select(0, idx)) if len(valid) else np.zeros((0, cfg.T, cfg.D), np.uint16)
    local = np.full(len(row), -1, dtype=np.int32)
    local[valid] = np.arange(len(valid), dtype=np.int32)
    local[P:] = -1
    if len(kp) == 0:  # keep a non-empty buffer for the oracle's pointer
        kp = np.zeros((1, cfg.T, cfg.D), np.uint16)
        vp = np.zeros((1, cfg.T, cfg.D), np.uint16)
    return kp, vp, local


def q_group(wl, q, b, h):
    G = wl.cfg.G
    return bf16_bits(q[b, h * G:(h + 1) * G])


def check_selection(s_gpu, s_orc, sel_gpu, K, stats: Stats):
    """The GPU selection against its own scores (exact) and the oracle's (tie window)."""
    P = len(s_orc)
    assert np.all(np.abs(s_gpu - s_orc) <= SCORE_RTOL * max(np.abs(s_orc).max(), 1e-30)), \
        f"scores differ by {np.abs(s_gpu - s_orc).max():.3e}"
    own = oracle.topk(s_gpu, K)
    assert sel_gpu.tolist() == own.tolist(), "GPU selection is not the top-K of its own scores"
    ref = oracle.topk(s_orc, K)
    n = min(K, P)
    s_k = np.sort(s_orc)[::-1][n - 1]
    for p in set(sel_gpu.tolist()) ^ set(ref.tolist()):
        assert abs(s_orc[p] - s_k) <= TIE_RTOL * max(abs(s_k), 1e-30), \
            f"page {p} selected differently (score {s_orc[p]!r}, K-th {s_k!r})"
        stats.ties += 1


def check_selection_vs_oracle(s_orc, sel_gpu, K, stats: Stats):
    """The GPU selection against the oracle's, without the GPU's scores: the two may differ only on pages
    whose oracle score lies within the tie window of the oracle's K-th score (each such page is counted).
    The selection must still be ascending, distinct and min(K, P) long."""
    P = len(s_orc)
    n = min(K, P)
    sel = [int(x) for x in sel_gpu]
    assert len(sel) == n, f"{len(sel)} pages selected, want {n}"
    assert all(a < b for a, b in zip(sel, sel[1:])), "selection not strictly ascending"
    assert all(0 <= x < P for x in sel), "selected page out of range"
    if n == 0:
        return
    ref = oracle.topk(s_orc, K)
    s_k = np.sort(s_orc)[::-1][n - 1]
    for p in set(sel) ^ set(ref.tolist()):
        assert abs(s_orc[p] - s_k) <= TIE_RTOL * max(abs(s_k), 1e-30), \
            f"page {p} selected differently (score {s_orc[p]!r}, K-th {s_k!r})"
        stats.ties += 1


def compare_attention(out_gpu, lse_gpu, out_ref, lse_ref, stats: Stats):
    out_gpu = np.asarray(out_gpu, dtype=np.float64)
    d = np.abs(out_gpu - out_ref)
    stats.max_abs = max(stats.max_abs, float(d.max()) if d.size else 0.0)
    stats.abs_err_sum += float(d.sum())
    stats.ref_abs_sum += float(np.abs(out_ref).sum())
    finite = np.isfinite(lse_ref)
    assert np.array_equal(finite, np.isfinite(lse_gpu)), "lse -inf pattern differs"
    if finite.any():
        stats.lse_max_abs = max(stats.lse_max_abs, float(np.abs(lse_gpu[finite] - lse_ref[finite]).max()))


def check_unit(wl, st, layer, b, h, q, scores_gpu=None, stats: Stats | None = None, full=None,
               check_meta=True, group_reduce=0, sel_vs_oracle=False):
    """Compare one unit of one layer (after select + attend) with the oracle.  With ``scores_gpu`` the
    selection is checked against the GPU's own scores and the oracle's; without them, ``sel_vs_oracle``
    checks it against the oracle's selection from ``q`` (for a unit selected in this step)."""
    stats = stats or Stats()
    cfg = wl.cfg
    G, T = cfg.G, cfg.T
    seq = int(wl.seq_len[b])
    P = -(-seq // T)
    kp, vp, row = unit_pool(wl, b, layer, h, full)
    meta_o, err = oracle.unit_minmax(kp, T, row, seq)
    if check_meta:
        meta_g = bf16_bits(st.meta[b, layer, h, :P])
        assert np.array_equal(meta_o[:P], meta_g), "MinMax metadata differs"
    qg = q_group(wl, q, b, h)
    cnt = int(st.sel_cnt[b, layer, h])
    sel_g = st.sel_idx[b, layer, h, :cnt].cpu().numpy()
    if scores_gpu is not None:
        s_o = oracle.unit_scores(qg, meta_o, P, group_reduce)
        s_g = scores_gpu[b, h, :P].double().cpu().numpy()
        check_selection(s_g, s_o, sel_g, st.K, stats)
    elif sel_vs_oracle:
        check_selection_vs_oracle(oracle.unit_scores(qg, meta_o, P, group_reduce), sel_g, st.K, stats)
    out_o, lse_o, _ = oracle.unit_sparse_attention(qg, kp, vp, T, row, seq, sel_g)
    out_g = st.out[layer, b, h * G:(h + 1) * G].cpu().numpy()
    lse_g = st.lse[layer, b, h * G:(h + 1) * G].cpu().numpy()
    compare_attention(out_g, lse_g, out_o, lse_o, stats)
    stats.units += 1
    return stats
