"""Full-size workloads on the GPU, checked on sampled units against the oracle.

Every configuration runs at its real shape with automatic split counts, as
the benchmark launches it; a spread of units (batch, layer, KV head) is pulled
to the host and compared with the oracle (metadata bit-exact, selection
within the tie window, attention within 2e-3 max-abs / 1e-3 mean-relative).
The wide-GQA configuration allocates 8 of its 64 layers, like the benchmark.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from paged_kv_cache_minmax_gb300.workloads import CONFIGS, bf16_bits
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from paged_kv_cache_minmax_gb300 import build

    build.build_library()
    kvmm.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def sample_units(cfg, n, seed):
    rs = np.random.default_rng(seed)
    units = {(0, 0, 0), (cfg.B - 1, cfg.L_alloc - 1, cfg.Hkv - 1)}
    while len(units) < n:
        units.add((int(rs.integers(cfg.B)), int(rs.integers(cfg.L_alloc)), int(rs.integers(cfg.Hkv))))
    return sorted(units)


@pytest.mark.parametrize("cfg_id", [2, 3, 5])
def test_fullsize_decode_step_sampled(cfg_id):
    cfg = CONFIGS[cfg_id]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    units = sample_units(cfg, 8, cfg.seed)
    layers = sorted({l for _, l, _ in units})
    nk, nv = workloads.step_tokens(wl, 0)
    scores = {}
    for l in range(cfg.L_alloc):
        s = torch.zeros(cfg.B, cfg.Hkv, cfg.Pmax, device="cuda") if l in layers else None
        st.append(l, nk[l], nv[l])  # the current token lands at position seq_len - 1
        st.select(l, wl.q[l], scores_out=s)
        st.diff(l)
        st.attend(l, wl.q[l])
        scores[l] = s
    torch.cuda.synchronize()
    assert st.read_err() == 0
    stats = parity.Stats()
    for (b, l, h) in units:
        parity.check_unit(wl, st, l, b, h, wl.q[l], scores[l], stats)
    stats.check()
    # the planted pages lead the selection
    b, l, h = units[0]
    pl = set(wl.planted[b, l, h].tolist())
    sel = set(st.sel_idx[b, l, h, : int(st.sel_cnt[b, l, h])].tolist())
    assert len(pl & sel) >= 0.7 * min(len(pl), cfg.K)  # MinMax bounds are noisy estimators
    print(cfg.name, "units", stats.units, "ties", stats.ties, "max-abs", stats.max_abs,
          "mean-rel", stats.mean_rel)


def test_fullsize_stable_unstable_drift_sampled():
    """Config 4 at full size: 64 steps, 25% unstable heads, rerank every 16 steps."""
    cfg = CONFIGS[4]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    qs = workloads.drift_queries(wl, cfg.steps)
    unstable = wl.unstable.cpu().numpy()
    units = sample_units(cfg, 6, 44)
    # include one unstable and one stable head
    l_u, h_u = map(int, np.argwhere(unstable == 1)[0])
    l_s, h_s = map(int, np.argwhere(unstable == 0)[0])
    units = sorted(set(units) | {(1, l_u, h_u), (2, l_s, h_s)})
    check_steps = {0, 1, 15, 16, 17, 40, 63}
    prev_sel = {u: None for u in units}
    promoted_log = []
    for step in range(cfg.steps):
        nk, nv = workloads.step_tokens(wl, step)
        wl.seq_len += 1
        resc = np.array([[oracle.rescored(unstable[l, h], step, cfg.rerank_period) for h in range(cfg.Hkv)]
                         for l in range(cfg.L)], dtype=np.uint8)
        mask = torch.as_tensor(resc, device="cuda")
        want = {l for _, l, _ in units} if step in check_steps else set()
        sc = {}
        for l in range(cfg.L):
            s = torch.zeros(cfg.B, cfg.Hkv, cfg.Pmax, device="cuda") if l in want else None
            st.append(l, nk[l], nv[l])
            st.select(l, qs[step, l], rescore_mask=mask, scores_out=s)
            st.diff(l, rescore_mask=mask)
            st.attend(l, qs[step, l])
            sc[l] = s
        promoted_log.append(int(st.promoted_cnt.sum()))
        torch.cuda.synchronize()
        assert st.read_err() == 0
        stats = parity.Stats()
        for (b, l, h) in units:
            cnt = int(st.sel_cnt[b, l, h])
            sel = st.sel_idx[b, l, h, :cnt].tolist()
            if not resc[l, h]:
                assert sel == prev_sel[(b, l, h)] and int(st.promoted_cnt[b, l, h]) == 0
            else:
                n_p = int(st.promoted_cnt[b, l, h])
                base = prev_sel[(b, l, h)] or []
                assert st.promoted[b, l, h, :n_p].tolist() == sorted(set(sel) - set(base))
            if step in check_steps:
                parity.check_unit(wl, st, l, b, h, qs[step, l], sc[l] if resc[l, h] else None, stats)
            prev_sel[(b, l, h)] = sel
        if step in check_steps:
            stats.check()
    # stable heads promote only on rerank steps; unstable ones may promote every step
    assert promoted_log[16] > 0
    print("promoted per step", promoted_log)
