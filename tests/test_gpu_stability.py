"""GPU parity of topk_history_record and topk_stability_rco (head stability profiling).

FlexiCache blog summary (MLSys'26), "Core insight: attention heads differ in
temporal stability": per-head top-K sets recorded over a window, compared a
few steps apart with the Random-Corrected Overlap, the least stable quarter of
the heads classed unstable.  The kernels must reproduce the oracle's per-unit
RCO means (float32 of the oracle's double), its per-head means over the batch
and its classification, on random ragged histories that wrap around the ring;
and profiling a workload whose unstable heads' queries drift fast must find
exactly those heads.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState, StabilityProfiler

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from paged_kv_cache_minmax_gb300 import build

    build.build_library()
    kvmm.load()
    oracle.build()
    yield
    torch.cuda.empty_cache()


def oracle_expectations(steps, B, L, Hkv, W, n, lag, frac):
    """rco per unit (float32), stability per head (float32) and the mask, from the recorded steps (host)."""
    newest = len(steps) - 1
    window = [steps[newest - t] for t in range(n)]  # newest first
    rco = np.zeros((B, L, Hkv), dtype=np.float32)
    for b in range(B):
        for l in range(L):
            for h in range(Hkv):
                idx = np.stack([st["idx"][b, l, h] for st in window])
                cnt = np.array([st["cnt"][b, l, h] for st in window], dtype=np.int32)
                pages = np.array([st["pages"][b] for st in window], dtype=np.int32)
                rco[b, l, h] = np.float32(oracle.unit_stability(idx, cnt, pages, lag))
    stab = np.zeros((L, Hkv), dtype=np.float64)
    for l in range(L):
        for h in range(Hkv):
            s = 0.0
            for b in range(B):
                s += float(rco[b, l, h])
            stab[l, h] = s / B
    mask = oracle.classify(stab, np.float32(frac)).reshape(L, Hkv)
    return rco, stab.astype(np.float32), mask


@pytest.mark.parametrize("lag,n", [(1, 7), (2, 7), (3, 5)])
def test_rco_and_classification_match_the_oracle(lag, n):
    B, L, Hq, Hkv, D, T, Pmax, Kmax, W = 2, 3, 8, 4, 64, 16, 40, 16, 7
    shape = kvmm.make_shape(B, L, Hq, Hkv, D, T, Pmax, Kmax, B * L * Hkv * Pmax)
    rng = np.random.default_rng(100 + lag)
    hist_idx = torch.full((W, B, L, Hkv, Kmax), -7, dtype=torch.int32, device="cuda")
    hist_cnt = torch.zeros(W, B, L, Hkv, dtype=torch.int32, device="cuda")
    hist_pages = torch.zeros(W, B, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    seq = rng.integers(1, Pmax * T // 2, size=B)
    steps = []
    for s in range(11):  # more steps than slots: the ring wraps
        seq = np.minimum(seq + rng.integers(0, 3 * T, size=B), Pmax * T)
        pages = -(-seq // T)
        idx = np.full((B, L, Hkv, Kmax), -1, dtype=np.int32)
        cnt = np.zeros((B, L, Hkv), dtype=np.int32)
        for b in range(B):
            for l in range(L):
                for h in range(Hkv):
                    top = min(Kmax, int(pages[b]))
                    c = top if rng.random() < 0.7 else int(rng.integers(0, top + 1))
                    pool = np.arange(int(pages[b]))
                    if rng.random() < 0.5 and steps:  # keep part of the previous selection
                        prev = steps[-1]["idx"][b, l, h][:steps[-1]["cnt"][b, l, h]]
                        keep = prev[rng.random(len(prev)) < 0.6]
                        rest = np.setdiff1d(pool, keep)
                        extra = rng.choice(rest, max(0, min(c - len(keep), len(rest))), replace=False)
                        sel = np.union1d(keep[:c], extra)[:c]
                    else:
                        sel = np.sort(rng.choice(pool, c, replace=False))
                    cnt[b, l, h] = len(sel)
                    idx[b, l, h, :len(sel)] = np.sort(sel)
        steps.append({"idx": idx, "cnt": cnt, "pages": pages.astype(np.int32)})
        d_idx = torch.tensor(idx, device="cuda")
        d_cnt = torch.tensor(cnt, device="cuda")
        d_seq = torch.tensor(seq.astype(np.int32), device="cuda")
        for l in range(L):
            kvmm.topk_history_record(shape, l, d_idx, d_cnt, d_seq, s % W, hist_idx, hist_cnt, hist_pages, err=err)
    head = (len(steps) - 1) % W
    rco = torch.zeros(B, L, Hkv, dtype=torch.float32, device="cuda")
    stab = torch.zeros(L, Hkv, dtype=torch.float32, device="cuda")
    mask = torch.zeros(L, Hkv, dtype=torch.uint8, device="cuda")
    kvmm.topk_stability_rco(shape, hist_idx, hist_cnt, hist_pages, n, head, lag, rco, stab, mask, 0.25, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_rco, want_stab, want_mask = oracle_expectations(steps, B, L, Hkv, W, n, lag, 0.25)
    np.testing.assert_array_equal(rco.cpu().numpy(), want_rco)
    np.testing.assert_array_equal(stab.cpu().numpy(), want_stab)
    np.testing.assert_array_equal(mask.cpu().numpy(), want_mask)
    assert int(mask.sum()) == round(0.25 * L * Hkv)


def test_out_of_range_history_is_reported_and_clamped():
    B, L, Hq, Hkv, D, T, Pmax, Kmax, W = 1, 1, 2, 2, 64, 16, 8, 4, 3
    shape = kvmm.make_shape(B, L, Hq, Hkv, D, T, Pmax, Kmax, 64)
    hist_idx = torch.arange(W * B * L * Hkv * Kmax, dtype=torch.int32, device="cuda").view(W, B, L, Hkv, Kmax) % 8
    hist_idx = hist_idx.sort(dim=-1).values.contiguous()
    hist_cnt = torch.full((W, B, L, Hkv), 2, dtype=torch.int32, device="cuda")
    hist_pages = torch.full((W, B), 8, dtype=torch.int32, device="cuda")
    rco = torch.zeros(B, L, Hkv, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvmm.topk_stability_rco(shape, hist_idx, hist_cnt, hist_pages, 3, 2, 1, rco, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hist_cnt[1, 0, 0, 1] = Kmax + 5
    hist_pages[2, 0] = Pmax + 1
    kvmm.topk_stability_rco(shape, hist_idx, hist_cnt, hist_pages, 3, 2, 1, rco, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvmm.ERR_OUT_OF_RANGE
    assert torch.isfinite(rco).all()
    # recording a sequence longer than the page table
    err.zero_()
    sel = torch.zeros(B, L, Hkv, Kmax, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, L, Hkv, dtype=torch.int32, device="cuda")
    seq = torch.tensor([Pmax * T + 1], dtype=torch.int32, device="cuda")
    kvmm.topk_history_record(shape, 0, sel, cnt, seq, 0, hist_idx, hist_cnt, hist_pages, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) & kvmm.ERR_OUT_OF_RANGE
    assert int(hist_pages[0, 0]) == Pmax


def test_profiling_finds_the_heads_whose_queries_drift():
    cfg = workloads.Config("stability", B=2, L=2, Hq=32, Hkv=8, D=128, T=16, S=8192, K=32, key_dist="outlier",
                           n_planted=32, unstable_frac=0.25, seed=91)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    W = 8
    qs = workloads.drift_queries_by_stability(wl, W)
    prof = StabilityProfiler(st.shape, W)
    for t in range(W):
        for l in range(cfg.L):
            st.select(l, qs[t][l])
        prof.record(st)
    rco, stab, mask = prof.classify(lag=1, unstable_frac=0.25)
    torch.cuda.synchronize()
    assert st.read_err() == 0 and int(prof.err.item()) == 0
    assert torch.equal(mask.cpu(), wl.unstable.cpu()), (stab.cpu(), wl.unstable.cpu())
    # and the same numbers as the oracle on the recorded history
    steps = []
    hi, hc, hp = prof.hist_idx.cpu().numpy(), prof.hist_cnt.cpu().numpy(), prof.hist_pages.cpu().numpy()
    for s in range(W):
        steps.append({"idx": hi[s], "cnt": hc[s], "pages": hp[s]})
    want_rco, want_stab, want_mask = oracle_expectations(steps, cfg.B, cfg.L, cfg.Hkv, W, W, 1, 0.25)
    np.testing.assert_array_equal(rco.cpu().numpy(), want_rco)
    np.testing.assert_array_equal(mask.cpu().numpy(), want_mask)
    print("stable mean", float(stab[wl.unstable == 0].mean()), "unstable mean", float(stab[wl.unstable == 1].mean()))
