"""decode_layer against the oracle at the launch shapes the benchmark times.

Every workload runs at full size through ``bench.decode_step`` -- the very call
sequence bench.py captures and replays: all allocated layers' decode_layer
launches back to back with early cache reads (KVMM_DECODE_EARLY_READS), the
automatic launch shape (units per cluster, CTAs per cluster) and the promotion
diff on a side stream, in a CUDA graph replayed several times.  Sampled units
of several layers are then pulled to the host and compared with the oracle:
MinMax metadata bit-exact, the selection equal to the oracle's except for
counted ties within 1e-5 of the K-th score, attention within 2e-3 max-abs /
1e-3 mean-relative.  One sampled layer is launched once more with its scores
written out, so that its selection is also checked against its own fp32 scores
bit for bit.

The stable/unstable workload runs its drifting 64-step episode (one appended
token per step, every unit rescored every 16 steps, the unstable heads' units
in between) through the same graphs as the benchmark; units are checked at
steps on both sides of a rerank, the kept selections of stable heads must not
move between reranks, and the promoted lists must be the set differences.

When the environment names a file in KVMM_PARITY_RECORD, each workload's
figures (units checked, ties, max-abs, mean-rel, launch shape, the sources'
digest) are merged into it as JSON; bench.py reports that record.
"""
import json
import os

import numpy as np
import pytest
import torch

import bench
from paged_kv_cache_minmax_gb300 import build as kbuild
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from paged_kv_cache_minmax_gb300.workloads import CONFIGS
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _clean():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    kbuild.build_library()
    kvmm.load()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def sample_units(cfg, n, seed):
    """n (batch, layer, KV head) units: the first and last unit of the first and last layer, the rest random."""
    rs = np.random.default_rng(seed)
    L = cfg.L_alloc
    units = {(0, 0, 0), (cfg.B - 1, L - 1, cfg.Hkv - 1), (cfg.B - 1, 0, cfg.Hkv - 1), (0, L - 1, 0)}
    while len(units) < n:
        units.add((int(rs.integers(cfg.B)), int(rs.integers(L)), int(rs.integers(cfg.Hkv))))
    return sorted(units)


def record(workload, entry):
    path = os.environ.get("KVMM_PARITY_RECORD")
    if not path:
        return
    d = {}
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
    d[workload] = entry
    with open(path, "w") as f:
        json.dump(d, f, indent=1, sort_keys=True)


def launch_shape(st):
    return {"units_per_cluster": kvmm.decode_layer_units(st.shape), "cluster_ctas": kvmm.decode_layer_cluster(st.shape)}


def entry_for(stats, st, units, extra):
    return {"units_checked": stats.units, "ties": stats.ties, "max_abs": stats.max_abs, "mean_rel": stats.mean_rel,
            "lse_max_abs": stats.lse_max_abs, "launch_shape": launch_shape(st), "early_reads": True,
            "layers_checked": sorted({l for _, l, _ in units}), "sources": kbuild.source_digest(),
            "test": "tests/test_gpu_bench_shapes.py", **extra}


@pytest.mark.parametrize("cfg_id", [2, 3, 5])
def test_bench_step_matches_oracle(cfg_id):
    cfg = CONFIGS[cfg_id]
    L = cfg.L_alloc
    wl = workloads.generate(cfg, device="cuda", seed=bench.replica_seed(cfg, 0))
    st = DecodeState.for_workload(wl)
    shape = launch_shape(st)
    assert shape["cluster_ctas"] >= 1 and shape["units_per_cluster"] >= 1, "decode_layer falls back"
    st.build_metadata()
    nk, nv = workloads.step_tokens(wl, 0)
    st.tok_begin.copy_(wl.seq_len - 1)
    q = wl.q.clone()
    torch.cuda.synchronize()  # the set-up above ran on the default stream; the steps run on their own
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    forks = [torch.cuda.Event() for _ in range(L)]
    with torch.cuda.stream(stream):  # eager first (as the benchmark warms up), then the captured step
        bench.decode_step(st, "decode_layer", L, q, nk, nv, True, side, forks)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        bench.decode_step(st, "decode_layer", L, q, nk, nv, True, side, forks)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g.replay()
    stream.synchronize()
    assert st.read_err() == 0
    units = sample_units(cfg, 12, cfg.seed)
    stats = parity.Stats()
    for (b, l, h) in units:
        parity.check_unit(wl, st, l, b, h, q[l], None, stats, sel_vs_oracle=True)
    # one sampled layer again with its scores written out: the same selection, the top K of its own scores
    b0, l0, h0 = units[len(units) // 2]
    keep = st.sel_idx.clone()
    sc = torch.zeros(cfg.B, cfg.Hkv, cfg.Pmax, device="cuda")
    with torch.cuda.stream(stream):
        kvmm.decode_layer(st.shape, l0, q[l0], nk[l0], nv[l0], 1, st.tok_begin, st.seq_len, st.k_pool, st.v_pool,
                          st.block_table, st.meta, st.seq_len, None, st.K, st.sel_idx, st.sel_cnt, st.out[l0],
                          lse=st.lse[l0], err=st.err, workspace=st.workspace, scores_out=sc, early_reads=True)
    stream.synchronize()
    assert torch.equal(keep, st.sel_idx), "writing the scores out changed a selection"
    for bb in range(cfg.B):
        for hh in range(cfg.Hkv):
            if (bb, hh) in ((b0, h0), (0, 0), (cfg.B - 1, cfg.Hkv - 1)):
                parity.check_unit(wl, st, l0, bb, hh, q[l0], sc, stats)
    stats.check()
    # the planted pages lead the selection
    pl = set(wl.planted[0, 0, 0].tolist())
    sel = set(st.sel_idx[0, 0, 0, : int(st.sel_cnt[0, 0, 0])].tolist())
    assert len(pl & sel) >= 0.7 * min(len(pl), cfg.K)
    record(cfg.name, entry_for(stats, st, units, {"steps": 4, "layers_run": L}))
    print(cfg.name, shape, "units", stats.units, "ties", stats.ties, "max-abs", stats.max_abs, "mean-rel",
          stats.mean_rel)


def test_mix_episode_matches_oracle():
    """The stable/unstable workload's 64-step drifting episode through the benchmark's per-step graphs."""
    cfg = CONFIGS[4]
    L = cfg.L_alloc
    wl = workloads.generate(cfg, device="cuda", seed=bench.replica_seed(cfg, 0))
    st = DecodeState.for_workload(wl)
    shape = launch_shape(st)
    assert shape["cluster_ctas"] >= 1, "decode_layer falls back"
    st.build_metadata()
    ep = bench.MixEpisode(wl, st)
    stream, side = torch.cuda.Stream(), torch.cuda.Stream()
    forks = [torch.cuda.Event() for _ in range(L)]

    def run(t):
        bench.decode_step(st, "decode_layer", L, ep.q[t], ep.nk[t], ep.nv[t], True, side, forks, mask=ep.mask(t),
                          tok_begin=ep.tb[t], seq_len=ep.seq[t], total_promoted=ep.prom[t:t + 1])

    graphs = []
    for t in range(ep.E):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(t)
        graphs.append(g)
    st.prev_cnt.zero_()
    torch.cuda.synchronize()  # the set-up ran on the default stream; the steps run on their own
    unstable = ep.unstable.cpu().numpy()
    units = sample_units(cfg, 8, 44)
    l_u, h_u = map(int, np.argwhere(unstable == 1)[0])
    l_s, h_s = map(int, np.argwhere(unstable == 0)[0])
    units = sorted(set(units) | {(1, l_u, h_u), (2, l_s, h_s)})
    check_steps = {0, 1, 15, 16, 17, 40, 63}
    prev_sel = {u: [] for u in units}
    stats = parity.Stats()
    promoted = []
    for t in range(ep.E):
        with torch.cuda.stream(stream):
            graphs[t].replay()
        stream.synchronize()
        assert st.read_err() == 0, f"step {t}"
        promoted.append(int(st.promoted_cnt.sum()))
        assert int(ep.prom[t]) == promoted[-1], "total_promoted disagrees with the per-unit counts"
        wl.seq_len.copy_(ep.seq[t])
        for (b, l, h) in units:
            resc = ep.rerank(t) or unstable[l, h] == 1
            sel = st.sel_idx[b, l, h, : int(st.sel_cnt[b, l, h])].tolist()
            n_p = int(st.promoted_cnt[b, l, h])
            if not resc:
                assert sel == prev_sel[(b, l, h)] and n_p == 0, f"step {t}: a kept selection moved"
            else:
                assert st.promoted[b, l, h, :n_p].tolist() == sorted(set(sel) - set(prev_sel[(b, l, h)]))
            if t in check_steps:
                parity.check_unit(wl, st, l, b, h, ep.q[t, l], None, stats, sel_vs_oracle=bool(resc))
            prev_sel[(b, l, h)] = sel
    stats.check()
    assert promoted[16] > 0 and promoted[0] == cfg.B * L * cfg.Hkv * cfg.K
    record(cfg.name, entry_for(stats, st, units, {"steps": ep.E, "layers_run": L,
                                                  "checked_steps": sorted(check_steps)}))
    print(cfg.name, shape, "units", stats.units, "ties", stats.ties, "max-abs", stats.max_abs, "mean-rel",
          stats.mean_rel, "promoted per step", promoted)
