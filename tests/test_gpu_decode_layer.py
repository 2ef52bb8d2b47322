"""GPU parity of decode_layer (append, score, select and attend in one launch).

It must leave exactly what kv_minmax_update followed by page_score_topk_attn
leaves: the appended rows in the pools and their pages' MinMax bit-exact, the
scores, selections and counts bit-exact, and the attention within the
attention tolerance of the oracle (and within 2e-5 of the separate calls).
Cases cover both group reductions, every (D, T), an odd number of units (a
cluster with one unit), short and empty sequences, partial rescore masks,
null blocks and no append at all.
"""
import pytest
import torch

from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from paged_kv_cache_minmax_gb300.workloads import CONFIGS, scaled
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    from paged_kv_cache_minmax_gb300 import build

    build.build_library()
    kvmm.load()
    yield
    torch.cuda.empty_cache()


CASES = {
    "tiny": CONFIGS[1],
    "llama-ragged": scaled(CONFIGS[2], B=2, L=2, S=4096, K=32, n_planted=16, ragged=True),
    "odd-units": workloads.Config("odd", B=3, L=1, Hq=12, Hkv=3, D=128, T=16, S=2000, K=20, ragged=True, seed=81),
    "permuted": scaled(CONFIGS[3], B=2, L=1, S=8192 + 5, K=64, n_planted=32),
    "gqa5-t32": scaled(CONFIGS[5], B=2, L=2, S=4096 - 7, K=16, n_planted=8, ragged=True, layers_alloc=None),
    "d64-g8": workloads.Config("d64-g8", B=2, L=1, Hq=16, Hkv=2, D=64, T=16, S=1500, K=12, key_dist="chanscale",
                               n_planted=6, ragged=True, permuted_pool=True, seed=77),
    "d64-t32": workloads.Config("d64-t32", B=3, L=1, Hq=8, Hkv=2, D=64, T=32, S=3000, K=40, ragged=True, seed=79),
    "g1-d128-t32": workloads.Config("g1-d128", B=1, L=1, Hq=4, Hkv=4, D=128, T=32, S=777, K=5, seed=78),
    "big-k": scaled(CONFIGS[2], B=1, L=1, S=32768, K=1000, n_planted=64),
}


def twin_states(cfg, group_reduce=0):
    """Two identical workloads and states: one for decode_layer, one for the separate calls."""
    out = []
    for _ in range(2):
        wl = workloads.generate(cfg, device="cuda")
        st = DecodeState.for_workload(wl, group_reduce=group_reduce)
        st.build_metadata()
        out.append((wl, st))
    torch.cuda.synchronize()
    return out


def run_both(a, b, layer, q, nk=None, nv=None, mask=None):
    (wa, sa), (wb, sb) = a, b
    cfg = wa.cfg
    sca = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    scb = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    sa.decode(layer, q, nk, nv, rescore_mask=mask, scores_out=sca)
    if nk is not None:
        sb.append(layer, nk, nv)
    sb.select(layer, q, rescore_mask=mask, scores_out=scb)
    sb.attend(layer, q)
    torch.cuda.synchronize()
    return sca, scb


def assert_same(a, b, sca, scb, layer):
    (wa, sa), (wb, sb) = a, b
    assert torch.equal(wa.k_pool, wb.k_pool), "appended key rows differ"
    assert torch.equal(wa.v_pool, wb.v_pool), "appended value rows differ"
    assert torch.equal(sa.meta, sb.meta), "MinMax metadata differs"
    assert torch.equal(sa.sel_cnt, sb.sel_cnt)
    for idx in torch.nonzero(torch.ones_like(sa.sel_cnt)).tolist():
        n = int(sa.sel_cnt[tuple(idx)])
        assert torch.equal(sa.sel_idx[tuple(idx)][:n], sb.sel_idx[tuple(idx)][:n]), idx
    assert torch.equal(torch.nan_to_num(sca, nan=7.0), torch.nan_to_num(scb, nan=7.0)), "scores differ"
    d = (sa.out[layer] - sb.out[layer]).abs().max().item()
    assert d <= 2e-5, f"attention differs by {d}"
    fa, fb = torch.isfinite(sa.lse[layer]), torch.isfinite(sb.lse[layer])
    assert torch.equal(fa, fb)
    assert (sa.lse[layer][fa] - sb.lse[layer][fb]).abs().max().item() <= 2e-5 if fa.any() else True


@pytest.mark.parametrize("name", sorted(CASES))
def test_decode_layer_matches_separate_calls_and_oracle(name):
    cfg = CASES[name]
    a, b = twin_states(cfg)
    wl, st = a
    nk, nv = workloads.step_tokens(wl, 0)
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        sca, scb = run_both(a, b, l, wl.q[l], nk[l], nv[l])
        assert st.read_err() == 0 and b[1].read_err() == 0
        assert_same(a, b, sca, scb, l)
        for bb in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wl, st, l, bb, h, wl.q[l], sca, stats)
    stats.check()
    print(name, "units", stats.units, "ties", stats.ties, "max-abs", stats.max_abs)


def test_without_append_equals_page_score_topk_attn():
    cfg = CASES["llama-ragged"]
    a, b = twin_states(cfg)
    for l in range(cfg.L):
        sca, scb = run_both(a, b, l, a[0].q[l])
        assert a[1].read_err() == 0
        assert_same(a, b, sca, scb, l)


def test_group_max_mode():
    cfg = CASES["gqa5-t32"]
    a, b = twin_states(cfg, group_reduce=1)
    nk, nv = workloads.step_tokens(a[0], 1)
    for l in range(cfg.L_alloc):
        sca, scb = run_both(a, b, l, a[0].q[l], nk[l], nv[l])
        assert a[1].read_err() == 0
        assert_same(a, b, sca, scb, l)


def test_repeated_steps_and_partial_rescore_mask():
    cfg = CASES["llama-ragged"]
    a, b = twin_states(cfg)
    qs = workloads.drift_queries(a[0], 4)
    for step in range(4):
        mask = None
        if step % 2 == 1:
            mask = torch.zeros(cfg.L_alloc, cfg.Hkv, dtype=torch.uint8, device="cuda")
            mask[:, 1::3] = 1
        nk, nv = workloads.step_tokens(a[0], step)
        for l in range(cfg.L):
            sca, scb = run_both(a, b, l, qs[step][l], nk[l], nv[l], mask=mask)
            assert a[1].read_err() == 0
            assert_same(a, b, sca, scb, l)


def test_short_and_empty_units():
    cfg = workloads.Config("short", B=3, L=1, Hq=8, Hkv=2, D=128, T=16, S=40, K=8, seed=5)
    a, b = twin_states(cfg)
    for wl, st in (a, b):
        wl.seq_len.copy_(torch.tensor([40, 1, 0], dtype=torch.int32))
        st.build_metadata()
    nk, nv = workloads.step_tokens(a[0], 0)
    # no append for the empty sequence: decode without new tokens
    sca, scb = run_both(a, b, 0, a[0].q[0])
    assert a[1].read_err() == 0
    assert_same(a, b, sca, scb, 0)
    assert a[1].sel_cnt[:, 0].tolist() == [[3, 3], [1, 1], [0, 0]]
    assert torch.all(a[1].out[0, 2] == 0)
    assert torch.all(torch.isneginf(a[1].lse[0, 2]))


def test_null_blocks_outside_the_selection_are_never_read():
    cfg = CASES["llama-ragged"]
    a, b = twin_states(cfg)
    wl, st = a
    for l in range(cfg.L):
        st.decode(l, wl.q[l])
    torch.cuda.synchronize()
    ref = st.out.clone()
    sel_mask = torch.zeros(cfg.B, cfg.L, cfg.Hkv, cfg.Pmax, dtype=torch.bool, device="cuda")
    for bb in range(cfg.B):
        for l in range(cfg.L):
            for h in range(cfg.Hkv):
                n = int(st.sel_cnt[bb, l, h])
                sel_mask[bb, l, h, st.sel_idx[bb, l, h, :n].long()] = True
    wl.block_table.masked_fill_(~sel_mask, kvmm.NULL_BLOCK)
    for l in range(cfg.L):
        st.decode(l, wl.q[l])
    torch.cuda.synchronize()
    assert st.read_err() == 0
    assert torch.equal(st.out, ref)
    victim = int(st.sel_idx[0, 0, 0, 3])
    wl.block_table[0, 0, 0, victim] = kvmm.NULL_BLOCK
    st.decode(0, wl.q[0])
    torch.cuda.synchronize()
    assert st.read_err() & kvmm.ERR_NULL_BLOCK
    assert not st.read_err() & kvmm.ERR_TIMEOUT
    stats = parity.Stats()
    parity.check_unit(wl, st, 0, 0, 0, wl.q[0], None, stats, check_meta=False)
    stats.check()


@pytest.mark.parametrize("pages,K,clustered", [(8192, 96, True), (8192, 300, True), (6000, 300, True),
                                               (12288, 96, True), (16384, 1500, False)])
def test_launch_shape_and_long_units(pages, K, clustered):
    """decode_layer's launch shape is one the device can hold: two units a cluster at the 8B shape; for one
    long unit (6000 to 12288 pages) a cluster that selects in two levels, each CTA keeping the scores of its
    own share; and none at 16384 pages with K = 1500 (the candidates no longer fit), where decode_layer runs
    the append and page_score_topk_attn instead.  Either way it leaves what the separate calls leave.  At
    K = 300 the selection takes the general top-K path (more than 2048 scores) at one of its two levels."""
    bench_shape = kvmm.make_shape(8, 32, 32, 8, 128, 16, 2048, 128, 1)
    assert kvmm.decode_layer_units(bench_shape) == 2
    assert 1 <= kvmm.decode_layer_cluster(bench_shape) <= 16
    cfg = workloads.Config("long", B=1, L=1, Hq=4, Hkv=1, D=128, T=16, S=16 * pages - 3, K=K,
                           key_dist="outlier", n_planted=24, seed=83)
    a, b = twin_states(cfg)
    wl, st = a
    if clustered:
        assert kvmm.decode_layer_units(st.shape) == 1  # one unit: a one-unit layout
        c = kvmm.decode_layer_cluster(st.shape)
        assert c > 1  # two levels
        if K == 300:  # one level over more than 2048 scores: a CTA's share, or the cluster's candidates
            assert max((pages + c - 1) // c, c * K) > 2048
    else:
        assert kvmm.decode_layer_units(st.shape) == 0 and kvmm.decode_layer_cluster(st.shape) == 0
    nk, nv = workloads.step_tokens(wl, 0)
    sca, scb = run_both(a, b, 0, wl.q[0], nk[0], nv[0])
    assert st.read_err() == 0 and b[1].read_err() == 0
    assert_same(a, b, sca, scb, 0)
    stats = parity.Stats()
    parity.check_unit(wl, st, 0, 0, 0, wl.q[0], sca, stats)
    stats.check()
    # a step that rescores nothing keeps the selection (and skips the two-level exchange)
    keep = torch.zeros(cfg.L, cfg.Hkv, dtype=torch.uint8, device="cuda")
    before = st.sel_idx.clone()
    nk1, nv1 = workloads.step_tokens(wl, 1)
    sca, scb = run_both(a, b, 0, wl.q[0], nk1[0], nv1[0], mask=keep)
    assert st.read_err() == 0 and b[1].read_err() == 0
    assert torch.equal(st.sel_idx, before)
    assert_same(a, b, sca, scb, 0)


def test_two_level_launch_with_short_units():
    """Two-level selection is chosen per launch (Pmax above a CTA's register-path capacity), so the short units
    of a long launch select in two levels too: a unit of 151 pages over 16 CTAs (shares of 9 or 10 pages, each
    CTA's candidates its whole share), one of 51 pages and one of a single page (fewer pages than K: every
    page), beside a unit of 8192 pages.  decode_layer leaves what the separate calls leave, and each unit
    matches the oracle."""
    cfg = workloads.Config("mixed-long", B=4, L=1, Hq=4, Hkv=1, D=128, T=16, S=16 * 8192 - 3, K=96,
                           key_dist="outlier", n_planted=24, seed=85)
    lens = [16 * 8192 - 3, 150 * 16 + 7, 50 * 16 + 5, 1]
    out = []
    for _ in range(2):
        wl = workloads.generate(cfg, device="cuda")
        wl.seq_len.copy_(torch.tensor(lens, dtype=torch.int32, device="cuda"))
        st = DecodeState.for_workload(wl)
        st.build_metadata()
        out.append((wl, st))
    torch.cuda.synchronize()
    a, b = out
    wl, st = a
    assert kvmm.decode_layer_units(st.shape) == 1 and kvmm.decode_layer_cluster(st.shape) > 1  # two levels
    nk, nv = workloads.step_tokens(wl, 0)
    sca, scb = run_both(a, b, 0, wl.q[0], nk[0], nv[0])
    assert st.read_err() == 0 and b[1].read_err() == 0
    assert_same(a, b, sca, scb, 0)
    assert st.sel_cnt[:, 0, 0].tolist() == [96, 96, 51, 1]
    stats = parity.Stats()
    for bb in range(cfg.B):
        parity.check_unit(wl, st, 0, bb, 0, wl.q[0], sca, stats)
    stats.check()


EARLY_CASES = {
    "llama-6-layers": scaled(CONFIGS[2], B=4, L=6, S=4096, K=32, n_planted=16, ragged=True),
    "gqa5-t32": CASES["gqa5-t32"],
    "odd-units": scaled(CASES["odd-units"], L=3),
}


@pytest.mark.parametrize("name", sorted(EARLY_CASES))
def test_early_reads_leave_what_the_waiting_launch_leaves(name):
    """KVMM_DECODE_EARLY_READS: the layers' launches back to back on one stream, each streaming its metadata
    while the previous one drains, leave bit for bit what launches that wait for the previous one leave:
    pools, MinMax, selections, outputs.  Odd layers take their queries from a kernel that writes them just
    before the launch (the queries are read only after the wait), and the second step keeps the stable
    heads' selections (read after the wait as well)."""
    cfg = EARLY_CASES[name]
    runs = []
    for early in (True, False):
        wl = workloads.generate(cfg, device="cuda")
        st = DecodeState.for_workload(wl)
        st.build_metadata()
        nk, nv = workloads.step_tokens(wl, 0)
        st.tok_begin.copy_(st.seq_len - 1)
        qbuf = torch.empty_like(wl.q[0])
        mask = (wl.unstable != 0).to(torch.uint8)
        torch.cuda.synchronize()
        for step in range(2):
            for l in range(cfg.L_alloc):
                q = wl.q[l]
                if l % 2:
                    qbuf.copy_(q)
                    q = qbuf
                kvmm.decode_layer(st.shape, l, q, nk[l], nv[l], 1, st.tok_begin, st.seq_len, st.k_pool,
                                  st.v_pool, st.block_table, st.meta, st.seq_len, None if step == 0 else mask, st.K,
                                  st.sel_idx, st.sel_cnt, st.out[l], lse=st.lse[l], err=st.err,
                                  workspace=st.workspace, early_reads=early)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        runs.append((wl, st))
    (wa, sa), (wb, sb) = runs
    assert torch.equal(wa.k_pool, wb.k_pool) and torch.equal(wa.v_pool, wb.v_pool)
    assert torch.equal(sa.meta, sb.meta)
    assert torch.equal(sa.sel_cnt, sb.sel_cnt) and torch.equal(sa.sel_idx, sb.sel_idx)
    assert torch.equal(sa.out, sb.out)
    assert torch.equal(sa.lse, sb.lse)
    # and the waiting launches match the oracle
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        for bb in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wb, sb, l, bb, h, wb.q[l], None, stats, check_meta=False)
    stats.check()


@pytest.mark.parametrize("L", [2, 3])
def test_early_reads_across_growing_steps(L):
    """Decode steps of L layers back to back, every launch appending one token at the end of its
    sequences, so seq_len and tok_begin advance every step and the appends cross page boundaries.  Each
    step's inputs sit in buffers of their own, filled before the first launch: no other kernel runs between
    the launches, which form one chain of programmatic dependent launches.  A launch with early cache reads
    then reads the metadata row that the same layer's launch one step earlier wrote; that launch is L
    launches back, and only the launch just before may still run (every kvmm kernel lets the next one start
    after its own wait).  The early and the waiting runs leave the same bytes, step by step, and the
    waiting run matches the oracle."""
    steps = 24
    cfg = scaled(CONFIGS[2], B=4, L=L, S=4096 - 3, K=32, n_planted=16, ragged=True, steps=steps)
    runs = []
    for early in (True, False):
        wl = workloads.generate(cfg, device="cuda")
        st = DecodeState.for_workload(wl)
        st.build_metadata()
        qs = workloads.drift_queries(wl, steps)
        toks = [workloads.step_tokens(wl, t) for t in range(steps)]
        base = wl.seq_len.clone()
        seq = torch.stack([base + t + 1 for t in range(steps)]).contiguous()  # [steps, B]: after the append
        tb = (seq - 1).contiguous()
        outs = torch.zeros(steps, L, cfg.B, cfg.Hq, cfg.D, device="cuda")
        lses = torch.zeros(steps, L, cfg.B, cfg.Hq, device="cuda")
        torch.cuda.synchronize()
        for t in range(steps):
            nk, nv = toks[t]
            for l in range(L):
                kvmm.decode_layer(st.shape, l, qs[t, l], nk[l], nv[l], 1, tb[t], seq[t], st.k_pool, st.v_pool,
                                  st.block_table, st.meta, seq[t], None, st.K, st.sel_idx, st.sel_cnt, outs[t, l],
                                  lse=lses[t, l], err=st.err, workspace=st.workspace, early_reads=early)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        wl.seq_len.copy_(seq[-1])
        st.out.copy_(outs[-1])
        st.lse.copy_(lses[-1])
        runs.append((wl, st, outs, lses, qs))
    (wa, sa, oa, la, _), (wb, sb, ob, lb, qb) = runs
    assert torch.equal(wa.k_pool, wb.k_pool) and torch.equal(wa.v_pool, wb.v_pool)
    assert torch.equal(sa.meta, sb.meta)
    assert torch.equal(sa.sel_cnt, sb.sel_cnt) and torch.equal(sa.sel_idx, sb.sel_idx)
    for t in range(steps):
        assert torch.equal(oa[t], ob[t]), f"step {t}: outputs differ"
        assert torch.equal(la[t], lb[t]), f"step {t}: lse differs"
    stats = parity.Stats()
    for l in range(L):
        for bb in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wb, sb, l, bb, h, qb[-1, l], None, stats, sel_vs_oracle=True)
    stats.check()


@pytest.mark.parametrize("name", ["llama-6-layers", "gqa5-t32", "odd-units"])
def test_separate_calls_with_early_reads(name):
    """page_score_topk and sparse_paged_decode_attn (automatic launch shape) back to back for every layer over
    two steps with drifting queries, with KVMM_EARLY_READS on both (each launch's predecessor writes only
    selections, scores or outputs) and without: the same selections, scores and outputs bit for bit, and the
    waiting run matches the oracle."""
    cfg = EARLY_CASES[name]
    runs = []
    for early in (True, False):
        wl = workloads.generate(cfg, device="cuda")
        st = DecodeState.for_workload(wl)
        st.build_metadata()
        qs = workloads.drift_queries(wl, 2)
        sc = torch.zeros(2, cfg.L_alloc, cfg.B, cfg.Hkv, cfg.Pmax, device="cuda")
        outs = torch.zeros(2, cfg.L_alloc, cfg.B, cfg.Hq, cfg.D, device="cuda")
        torch.cuda.synchronize()
        for step in range(2):
            for l in range(cfg.L_alloc):
                kvmm.page_score_topk(st.shape, l, qs[step, l], st.meta, st.seq_len, None, st.K, st.sel_idx,
                                     st.sel_cnt, st.workspace, st.err, scores_out=sc[step, l], early_reads=early)
                kvmm.sparse_paged_decode_attn(st.shape, l, qs[step, l], st.k_pool, st.v_pool, st.block_table,
                                              st.seq_len, st.sel_idx, st.sel_cnt, outs[step, l], st.workspace,
                                              lse=st.lse[l], err=st.err, early_reads=early)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        st.out.copy_(outs[1])
        runs.append((wl, st, sc, outs, qs))
    (wa, sa, sca, oa, _), (wb, sb, scb, ob, qb) = runs
    assert torch.equal(sa.sel_cnt, sb.sel_cnt) and torch.equal(sa.sel_idx, sb.sel_idx)
    assert torch.equal(sca, scb)
    assert torch.equal(oa, ob)
    assert torch.equal(sa.lse, sb.lse)
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        for bb in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wb, sb, l, bb, h, qb[1, l], scb[1, l], stats)
    stats.check()
