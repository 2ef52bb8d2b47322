"""Decode-step driver over the four C-ABI calls.

:class:`DecodeState` owns the device buffers one long-context decode needs
beside the caller's pools (MinMax metadata, selections, the committed previous
selections, promotion lists, outputs, workspace, error word) and issues, per
layer and step, the calls in the method's order:

  1. ``kv_minmax_update``          append the new token, refresh its page's MinMax
  2. ``page_score_topk``           rescored units only (stable heads keep their top-K)
  3. ``topk_promotion_diff``       promoted = cur \\ prev (commit cur as prev)
  4. ``sparse_paged_decode_attn``  attention over the selected pages

or, with steps 2 and 4 in one launch, ``page_score_topk_attn`` then the diff.

(FlexiCache, "Core method", sections 1-3.)  Everything runs on one CUDA
stream; nothing here synchronises.
"""
from __future__ import annotations

import torch

from . import kvmm


class DecodeState:
    def __init__(self, B, L, Hq, Hkv, D, T, Pmax, K, k_pool, v_pool, block_table, seq_len, num_splits=0,
                 group_reduce=0, device="cuda"):
        self.shape = kvmm.make_shape(B, L, Hq, Hkv, D, T, Pmax, K, k_pool.shape[0])
        self.K = K
        self.num_splits = num_splits
        self.group_reduce = group_reduce
        self.k_pool, self.v_pool, self.block_table, self.seq_len = k_pool, v_pool, block_table, seq_len
        i32 = dict(dtype=torch.int32, device=device)
        self.meta = torch.zeros(B, L, Hkv, Pmax, 2, D, dtype=torch.bfloat16, device=device)
        self.sel_idx = torch.zeros(B, L, Hkv, K, **i32)
        self.sel_cnt = torch.zeros(B, L, Hkv, **i32)
        self.prev_idx = torch.zeros(B, L, Hkv, K, **i32)
        self.prev_cnt = torch.zeros(B, L, Hkv, **i32)
        self.promoted = torch.zeros(B, L, Hkv, K, **i32)
        self.promoted_cnt = torch.zeros(B, L, Hkv, **i32)
        self.evicted = torch.zeros(B, L, Hkv, K, **i32)
        self.evicted_cnt = torch.zeros(B, L, Hkv, **i32)
        self.total_promoted = torch.zeros(1, **i32)
        self.out = torch.zeros(L, B, Hq, D, dtype=torch.float32, device=device)
        self.lse = torch.zeros(L, B, Hq, dtype=torch.float32, device=device)
        self.err = torch.zeros(1, **i32)
        self.tok_begin = torch.zeros(B, **i32)
        self.tok_end = torch.zeros(B, **i32)
        self.workspace = kvmm.alloc_workspace(self.shape, num_splits, device=device)

    @classmethod
    def for_workload(cls, wl, K=None, **kw):
        c = wl.cfg
        return cls(c.B, c.L_alloc, c.Hq, c.Hkv, c.D, c.T, c.Pmax, K or c.K, wl.k_pool, wl.v_pool,
                   wl.block_table, wl.seq_len, **kw)

    # ------------------------------------------------------------------ #
    def build_metadata(self, layers=None) -> None:
        """Rebuild the MinMax of every page below seq_len (after a prefill)."""
        s = self.shape
        self.tok_begin.zero_()
        for l in (range(s.L) if layers is None else layers):
            kvmm.kv_minmax_update(s, l, None, None, 0, self.tok_begin, self.seq_len, self.k_pool, self.v_pool,
                                  self.block_table, self.meta, self.err)

    def append(self, layer, new_k, new_v) -> None:
        """Write one new token per batch entry at position seq_len-1 of ``layer``.

        new_k / new_v: ``[B, Hkv, 1, D]`` bf16; ``seq_len`` already counts the token.
        """
        torch.sub(self.seq_len, 1, out=self.tok_begin)
        kvmm.kv_minmax_update(self.shape, layer, new_k, new_v, 1, self.tok_begin, self.seq_len, self.k_pool,
                              self.v_pool, self.block_table, self.meta, self.err)

    def select(self, layer, q, rescore_mask=None, scores_out=None) -> None:
        kvmm.page_score_topk(self.shape, layer, q, self.meta, self.seq_len, rescore_mask, self.K, self.sel_idx,
                             self.sel_cnt, self.workspace, self.err, scores_out=scores_out,
                             group_reduce=self.group_reduce)

    def diff(self, layer, rescore_mask=None, commit=True) -> None:
        kvmm.topk_promotion_diff(self.shape, layer, rescore_mask, self.prev_idx, self.prev_cnt, self.sel_idx,
                                 self.sel_cnt, self.promoted, self.promoted_cnt, self.evicted, self.evicted_cnt,
                                 self.total_promoted, commit=commit, err=self.err)

    def attend(self, layer, q, sm_scale=0.0) -> None:
        kvmm.sparse_paged_decode_attn(self.shape, layer, q, self.k_pool, self.v_pool, self.block_table,
                                      self.seq_len, self.sel_idx, self.sel_cnt, self.out[layer], self.workspace,
                                      lse=self.lse[layer], err=self.err, sm_scale=sm_scale,
                                      num_splits=self.num_splits)

    def select_attend(self, layer, q, rescore_mask=None, scores_out=None, sm_scale=0.0) -> None:
        """select + attend in one launch (page_score_topk_attn)."""
        kvmm.page_score_topk_attn(self.shape, layer, q, self.meta, self.k_pool, self.v_pool, self.block_table,
                                  self.seq_len, rescore_mask, self.K, self.sel_idx, self.sel_cnt, self.out[layer],
                                  self.workspace, lse=self.lse[layer], err=self.err, scores_out=scores_out,
                                  group_reduce=self.group_reduce, sm_scale=sm_scale)

    def decode(self, layer, q, new_k=None, new_v=None, rescore_mask=None, scores_out=None, sm_scale=0.0) -> None:
        """decode_layer: append (new_k/new_v [B, Hkv, 1, D] at seq_len - 1), score, select, attend."""
        if new_k is not None:
            torch.sub(self.seq_len, 1, out=self.tok_begin)
        kvmm.decode_layer(self.shape, layer, q, new_k, new_v, 1, self.tok_begin, self.seq_len, self.k_pool,
                          self.v_pool, self.block_table, self.meta, self.seq_len, rescore_mask, self.K, self.sel_idx,
                          self.sel_cnt, self.out[layer], lse=self.lse[layer], err=self.err, scores_out=scores_out,
                          group_reduce=self.group_reduce, sm_scale=sm_scale, workspace=self.workspace)

    def layer_step(self, layer, q, new_k=None, new_v=None, rescore_mask=None, fused=True) -> None:
        """One layer of one decode step: append, select + attend, diff."""
        if new_k is not None:
            self.append(layer, new_k, new_v)
        if fused:
            self.select_attend(layer, q, rescore_mask)
            self.diff(layer, rescore_mask)
        else:
            self.select(layer, q, rescore_mask)
            self.diff(layer, rescore_mask)
            self.attend(layer, q)

    def read_err(self) -> int:
        return int(self.err.item())


class StabilityProfiler:
    """Offline profiling of head stability: a ring of the last W steps' selections of every (batch, layer,
    KV head) and the Random-Corrected Overlap classification (FlexiCache, "Core insight: attention heads
    differ in temporal stability").  ``record(state)`` stores one decode step of every layer; ``classify``
    returns (rco per unit [B, L, Hkv], stability [L, Hkv], unstable mask [L, Hkv])."""

    def __init__(self, shape, W: int, device="cuda"):
        s = shape
        i32 = dict(dtype=torch.int32, device=device)
        self.shape, self.W = s, W
        self.hist_idx = torch.zeros(W, s.B, s.L, s.Hkv, s.Kmax, **i32)
        self.hist_cnt = torch.zeros(W, s.B, s.L, s.Hkv, **i32)
        self.hist_pages = torch.zeros(W, s.B, **i32)
        self.rco_unit = torch.zeros(s.B, s.L, s.Hkv, dtype=torch.float32, device=device)
        self.stability = torch.zeros(s.L, s.Hkv, dtype=torch.float32, device=device)
        self.unstable = torch.zeros(s.L, s.Hkv, dtype=torch.uint8, device=device)
        self.err = torch.zeros(1, **i32)
        self.steps = 0

    def record(self, state, layers=None) -> None:
        """Store this step's selections of ``layers`` (default: all) in slot steps mod W, then advance."""
        slot = self.steps % self.W
        for l in [-1] if layers is None else layers:  # -1: every layer in one launch
            kvmm.topk_history_record(self.shape, l, state.sel_idx, state.sel_cnt, state.seq_len, slot,
                                     self.hist_idx, self.hist_cnt, self.hist_pages, err=self.err)
        self.steps += 1

    def classify(self, lag: int = 1, unstable_frac: float = 0.25, n: int | None = None):
        n = min(self.steps, self.W) if n is None else n
        kvmm.topk_stability_rco(self.shape, self.hist_idx, self.hist_cnt, self.hist_pages, n,
                                (self.steps - 1) % self.W, lag, self.rco_unit, self.stability, self.unstable,
                                unstable_frac, err=self.err)
        return self.rco_unit, self.stability, self.unstable
