"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Small shapes that span several 64-page score chunks, several attention tiles
per split and ragged tails are compared unit by unit in full; the edge cases
(all pages selected, null blocks, empty selections, signed zeros, split
counts, both group reductions, D = 64 and 128, T = 16 and 32, G = 1..8) each
have a case.  Full-size configurations live in ``test_gpu_fullsize.py``.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from paged_kv_cache_minmax_gb300.workloads import CONFIGS, bf16_bits, scaled
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


def host_pools(wl):
    return bf16_bits(wl.k_pool), bf16_bits(wl.v_pool)


def run_all_layers(wl, st, scores=True):
    cfg = wl.cfg
    sc = []
    for l in range(cfg.L_alloc):
        s = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda") if scores else None
        st.select(l, wl.q[l], scores_out=s)
        st.diff(l)
        st.attend(l, wl.q[l])
        sc.append(s)
    torch.cuda.synchronize()
    return sc


def check_all(wl, st, sc, full=None, group_reduce=0):
    cfg = wl.cfg
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        for b in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wl, st, l, b, h, wl.q[l], sc[l], stats, full=full, group_reduce=group_reduce)
    stats.check()
    return stats


SMALL = {
    "tiny": CONFIGS[1],
    "llama-ragged": scaled(CONFIGS[2], B=2, L=2, S=4096, K=32, n_planted=16, ragged=True),
    "permuted": scaled(CONFIGS[3], B=2, L=1, S=8192 + 5, K=64, n_planted=32),
    "gqa5-t32": scaled(CONFIGS[5], B=2, L=2, S=4096 - 7, K=16, n_planted=8, ragged=True, layers_alloc=None),
    "d64-g8": workloads.Config("d64-g8", B=2, L=1, Hq=16, Hkv=2, D=64, T=16, S=1500, K=12, key_dist="chanscale",
                               n_planted=6, ragged=True, permuted_pool=True, seed=77),
    "g1-d128": workloads.Config("g1-d128", B=1, L=1, Hq=4, Hkv=4, D=128, T=32, S=777, K=5, seed=78),
}


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_small_configs_match_oracle(name, splits):
    cfg = SMALL[name]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl, num_splits=splits)
    st.build_metadata()
    sc = run_all_layers(wl, st)
    assert st.read_err() == 0
    full = host_pools(wl) if wl.n_phys * cfg.T * cfg.D <= (1 << 24) else None
    stats = check_all(wl, st, sc, full=full)
    # the planted pages must dominate the selection (the workload is not arbitrary)
    if cfg.n_planted and cfg.key_dist != "chanscale":
        pl = set(wl.planted[0, 0, 0].tolist())
        sel = set(st.sel_idx[0, 0, 0, : int(st.sel_cnt[0, 0, 0])].tolist())
        assert len(pl & sel) >= min(len(pl), cfg.K) * 0.7  # MinMax bounds are noisy estimators
    print(name, splits, "ties", stats.ties, "max-abs", stats.max_abs, "mean-rel", stats.mean_rel)


def test_group_max_mode_matches_oracle():
    cfg = SMALL["llama-ragged"]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl, group_reduce=1)
    st.build_metadata()
    sc = run_all_layers(wl, st)
    assert st.read_err() == 0
    check_all(wl, st, sc, group_reduce=1)


def test_all_pages_selected_equals_dense_attention():
    """Tiny shape with K = P: sparse attention over every page is dense attention."""
    cfg = scaled(CONFIGS[1], K=64)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    run_all_layers(wl, st, scores=False)
    assert int(st.sel_cnt[0, 0, 0]) == 64
    assert st.sel_idx[0, 0, 0].tolist() == list(range(64))
    kp, vp = host_pools(wl)
    row = wl.block_table[0, 0, 0].cpu().numpy()
    qg = parity.q_group(wl, wl.q[0], 0, 0)
    dense, lse_d, _ = oracle.unit_dense_attention(qg, kp, vp, cfg.T, row, cfg.S)
    stats = parity.Stats()
    parity.compare_attention(st.out[0, 0].cpu().numpy(), st.lse[0, 0].cpu().numpy(), dense, lse_d, stats)
    stats.check()


def test_split_count_invariance():
    cfg = SMALL["llama-ragged"]
    wl = workloads.generate(cfg, device="cuda")
    outs = []
    for splits in (1, 2, 4, 8, 32, 0):  # explicit counts: one unit a cluster; 0: the clustered kernel
        st = DecodeState.for_workload(wl, num_splits=splits)
        st.build_metadata()
        run_all_layers(wl, st, scores=False)
        assert st.read_err() == 0
        outs.append((st.out.clone(), st.lse.clone()))
    for o, l in outs[1:]:
        assert torch.allclose(o, outs[0][0], rtol=0, atol=2e-5)
        assert torch.allclose(l, outs[0][1], rtol=0, atol=2e-5)


def test_null_blocks_are_never_read():
    cfg = SMALL["llama-ragged"]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    run_all_layers(wl, st, scores=False)
    ref_out = st.out.clone()
    # evict every unselected page: the table keeps its shape, entries become null
    sel_mask = torch.zeros(cfg.B, cfg.L, cfg.Hkv, cfg.Pmax, dtype=torch.bool, device="cuda")
    for b in range(cfg.B):
        for l in range(cfg.L):
            for h in range(cfg.Hkv):
                n = int(st.sel_cnt[b, l, h])
                sel_mask[b, l, h, st.sel_idx[b, l, h, :n].long()] = True
    wl.block_table.masked_fill_(~sel_mask, kvmm.NULL_BLOCK)
    for l in range(cfg.L):
        st.attend(l, wl.q[l])
    torch.cuda.synchronize()
    assert st.read_err() == 0
    assert torch.equal(st.out, ref_out)
    # a selected page mapped to the null block is reported and skipped
    victim = int(st.sel_idx[0, 0, 0, 3])
    wl.block_table[0, 0, 0, victim] = kvmm.NULL_BLOCK
    st.attend(0, wl.q[0])
    torch.cuda.synchronize()
    assert st.read_err() & kvmm.ERR_NULL_BLOCK
    stats = parity.Stats()
    parity.check_unit(wl, st, 0, 0, 0, wl.q[0], None, stats, check_meta=False)
    stats.check()
    # out-of-range physical id
    st.err.zero_()
    wl.block_table[0, 0, 0, victim] = wl.n_phys + 5
    st.attend(0, wl.q[0])
    torch.cuda.synchronize()
    assert st.read_err() & kvmm.ERR_OUT_OF_RANGE


def test_budget_covers_short_sequences_and_empty_units():
    cfg = workloads.Config("short", B=3, L=1, Hq=8, Hkv=2, D=128, T=16, S=40, K=8, seed=5)
    wl = workloads.generate(cfg, device="cuda")
    wl.seq_len.copy_(torch.tensor([40, 1, 0], dtype=torch.int32))
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    sc = run_all_layers(wl, st)
    assert st.read_err() == 0
    assert st.sel_cnt[:, 0].tolist() == [[3, 3], [1, 1], [0, 0]]
    assert st.sel_idx[0, 0, 0, :3].tolist() == [0, 1, 2]
    stats = parity.Stats()
    for b in range(2):
        for h in range(2):
            parity.check_unit(wl, st, 0, b, h, wl.q[0], sc[0], stats)
    stats.check()
    assert torch.all(st.out[0, 2] == 0)
    assert torch.all(torch.isneginf(st.lse[0, 2]))


def test_signed_zero_and_exact_ties_in_metadata_and_selection():
    cfg = workloads.Config("ties", B=1, L=1, Hq=4, Hkv=1, D=64, T=16, S=64 * 16, K=7, seed=9)
    wl = workloads.generate(cfg, device="cuda")
    # pages 10..29 identical and shifted along sign(sum of the group's queries):
    # identical, best scores -> the lowest indices win the ties
    direction = torch.sign(wl.q[0, 0].float().sum(0))
    wl.k_pool[10:30] = (wl.k_pool[10].float() + 3.0 * direction).to(torch.bfloat16)
    wl.k_pool[3, :, 0] = 0.0
    wl.k_pool[3, ::2, 0] = -0.0
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    sc = run_all_layers(wl, st)
    sel = st.sel_idx[0, 0, 0].tolist()
    assert sel == list(range(10, 17)), sel
    stats = parity.Stats()
    parity.check_unit(wl, st, 0, 0, 0, wl.q[0], sc[0], stats, full=host_pools(wl))
    stats.check()


def test_append_updates_pages_and_metadata_incrementally():
    cfg = scaled(SMALL["gqa5-t32"], S=300, steps=70, K=6, n_planted=0, ragged=False)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    kp, vp = host_pools(wl)
    rows = {(b, l, h): wl.block_table[b, l, h].cpu().numpy() for b in range(cfg.B) for l in range(cfg.L_alloc)
            for h in range(cfg.Hkv)}
    for step in range(cfg.steps):
        nk, nv = workloads.step_tokens(wl, step)
        wl.seq_len += 1
        for l in range(cfg.L_alloc):
            st.append(l, nk[l], nv[l])
        seq = int(wl.seq_len[0])
        for (b, l, h), row in rows.items():
            oracle.unit_append(kp, vp, cfg.T, row, seq - 1, seq, bf16_bits(nk[l, b, h]), bf16_bits(nv[l, b, h]))
    torch.cuda.synchronize()
    assert st.read_err() == 0
    assert np.array_equal(bf16_bits(wl.k_pool), kp) and np.array_equal(bf16_bits(wl.v_pool), vp)
    for (b, l, h), row in rows.items():
        seq = int(wl.seq_len[b])
        P = -(-seq // cfg.T)
        meta_o, _ = oracle.unit_minmax(kp, cfg.T, row, seq)
        assert np.array_equal(meta_o[:P], bf16_bits(st.meta[b, l, h, :P]))


def test_promotion_diff_matches_set_difference():
    cfg = workloads.Config("diff", B=2, L=2, Hq=8, Hkv=2, D=64, T=16, S=2000, K=40, seed=11)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    gen = torch.Generator(device="cpu").manual_seed(3)
    P = cfg.P
    prev_lists, cur_lists = {}, {}
    for b in range(cfg.B):
        for l in range(cfg.L):
            for h in range(cfg.Hkv):
                n1, n2 = [int(x) for x in torch.randint(0, cfg.K + 1, (2,), generator=gen)]
                if (b, l, h) == (0, 0, 0):
                    n1 = n2 = cfg.K  # identical lists
                a = torch.randperm(P, generator=gen)[:n1].sort().values
                c = a if (b, l, h) == (0, 0, 0) else torch.randperm(P, generator=gen)[:n2].sort().values
                st.prev_idx[b, l, h, :n1] = a.to(torch.int32).cuda()
                st.prev_cnt[b, l, h] = n1
                st.sel_idx[b, l, h, :len(c)] = c.to(torch.int32).cuda()
                st.sel_cnt[b, l, h] = len(c)
                prev_lists[(b, l, h)], cur_lists[(b, l, h)] = a.tolist(), c.tolist()
    mask = torch.tensor([[1, 0], [1, 1]], dtype=torch.uint8, device="cuda")
    total = 0
    for l in range(cfg.L):
        st.diff(l, rescore_mask=mask)  # [L, Hkv]: entry [l, h] decides unit (b, l, h)
    torch.cuda.synchronize()
    assert st.read_err() == 0
    for (b, l, h), a in prev_lists.items():
        c = cur_lists[(b, l, h)]
        rescored = bool(mask[l, h])
        n = int(st.promoted_cnt[b, l, h])
        m = int(st.evicted_cnt[b, l, h])
        if not rescored:
            assert n == 0 and m == 0
            assert st.prev_idx[b, l, h, : len(a)].tolist() == a  # not committed
            continue
        assert st.promoted[b, l, h, :n].tolist() == oracle.set_difference(c, a).tolist()
        assert st.evicted[b, l, h, :m].tolist() == oracle.set_difference(a, c).tolist()
        assert st.prev_idx[b, l, h, : len(c)].tolist() == c and int(st.prev_cnt[b, l, h]) == len(c)
        total += n
    assert int(st.total_promoted) == total


def test_drift_with_stable_and_unstable_heads():
    """Config-4 schedule, scaled: unstable heads rescore every step, stable ones every 16."""
    cfg = scaled(CONFIGS[4], B=2, L=2, Hq=16, Hkv=4, S=2048, K=16, n_planted=8, steps=20)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    qs = workloads.drift_queries(wl, cfg.steps)
    kp, vp = host_pools(wl)
    units = [(b, l, h) for b in range(cfg.B) for l in range(cfg.L) for h in range(cfg.Hkv)]
    rows = {u: wl.block_table[u].cpu().numpy() for u in units}
    unstable = wl.unstable.cpu().numpy()
    assert unstable.sum() == 2
    prev_sel = {u: [] for u in units}
    promoted_total = 0
    for step in range(cfg.steps):
        nk, nv = workloads.step_tokens(wl, step)
        wl.seq_len += 1
        resc = np.array([[oracle.rescored(unstable[l, h], step, cfg.rerank_period) for h in range(cfg.Hkv)]
                         for l in range(cfg.L)], dtype=np.uint8)
        mask = torch.as_tensor(resc, device="cuda")
        sc = []
        for l in range(cfg.L):
            s = torch.zeros(cfg.B, cfg.Hkv, cfg.Pmax, device="cuda")
            st.append(l, nk[l], nv[l])
            st.select(l, qs[step, l], rescore_mask=mask, scores_out=s)
            st.diff(l, rescore_mask=mask)
            st.attend(l, qs[step, l])
            sc.append(s)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        seq = int(wl.seq_len[0])
        stats = parity.Stats()
        for (b, l, h) in units:
            oracle.unit_append(kp, vp, cfg.T, rows[(b, l, h)], seq - 1, seq, bf16_bits(nk[l, b, h]),
                               bf16_bits(nv[l, b, h]))
        for (b, l, h) in units:
            cnt = int(st.sel_cnt[b, l, h])
            sel = st.sel_idx[b, l, h, :cnt].tolist()
            n_p = int(st.promoted_cnt[b, l, h])
            if resc[l, h]:
                parity.check_unit(wl, st, l, b, h, qs[step, l], sc[l], stats, full=(kp, vp))
                assert st.promoted[b, l, h, :n_p].tolist() == sorted(set(sel) - set(prev_sel[(b, l, h)]))
                n_e = int(st.evicted_cnt[b, l, h])
                assert st.evicted[b, l, h, :n_e].tolist() == sorted(set(prev_sel[(b, l, h)]) - set(sel))
                promoted_total += n_p
            else:
                assert sel == prev_sel[(b, l, h)] and n_p == 0  # stable head reuses its top-K
                parity.check_unit(wl, st, l, b, h, qs[step, l], None, stats, full=(kp, vp))
            prev_sel[(b, l, h)] = sel
        stats.check()
    assert int(st.total_promoted) == promoted_total
