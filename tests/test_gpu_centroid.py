"""GPU parity of the centroid level of KVDrive's index (kv_centroid_build) and the two-level selection
(page_score_topk_centroid) against the oracle.

The build is compared bit for bit: centroids, assignments, member offsets and lists.  Its decisions are
taken on both sides in the same fp32 arithmetic and order.  The selection is checked in three ways:
  * the centroid scores within 1e-5 of the oracle's (fp32 against double);
  * the expanded pages exactly the members of the top M of the GPU's own centroid scores, and that top M
    equal to the oracle's but for centroids in the tie window;
  * the selected pages the exact top K of the GPU's own candidate scores, and equal to the oracle's top K
    over the same candidates but for counted ties.
Cases cover D 64/128, T 16/32, ragged and empty sequences, R from 1 to 8, no iteration (the spatial
blocking) to several, both group reductions, M beyond the centroid count, and a partial rescore mask.
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
    oracle.build()
    yield
    torch.cuda.empty_cache()


CASES = {
    "llama-ragged": scaled(CONFIGS[2], B=2, L=2, S=4096 + 5, K=32, n_planted=16, ragged=True),
    "gqa5-t32": scaled(CONFIGS[5], B=2, L=1, S=3000, K=16, n_planted=8, ragged=True, layers_alloc=None),
    "d64": workloads.Config("d64", B=3, L=1, Hq=8, Hkv=2, D=64, T=16, S=1500, K=12, key_dist="chanscale",
                            n_planted=6, ragged=True, permuted_pool=True, seed=91),
}


class Index:
    """A layer's mean keys and centroid index on the GPU."""

    def __init__(self, wl, st, R):
        c = wl.cfg
        self.R = R
        self.cmax = kvmm.centroid_rows(st.shape, R)
        dev = dict(device="cuda")
        self.mean = torch.zeros(c.B, c.L_alloc, c.Hkv, c.Pmax, c.D, dtype=torch.bfloat16, **dev)
        self.cent = torch.zeros(c.B, c.L_alloc, c.Hkv, self.cmax, c.D, dtype=torch.bfloat16, **dev)
        self.assign = torch.full((c.B, c.L_alloc, c.Hkv, c.Pmax), -3, dtype=torch.int32, **dev)
        self.off = torch.full((c.B, c.L_alloc, c.Hkv, self.cmax + 1), -3, dtype=torch.int32, **dev)
        self.members = torch.full((c.B, c.L_alloc, c.Hkv, c.Pmax), -3, dtype=torch.int32, **dev)
        for l in range(c.L_alloc):
            kvmm.kv_meankey_update(st.shape, l, None, wl.seq_len, wl.k_pool, wl.block_table, self.mean, err=st.err)

    def build(self, st, l, n_iter):
        kvmm.kv_centroid_build(st.shape, l, self.mean, st.seq_len, self.R, n_iter, self.cent, self.assign, self.off,
                               self.members, err=st.err)


def check_build(wl, idx, l, n_iter):
    c = wl.cfg
    for b in range(c.B):
        P = -(-int(wl.seq_len[b]) // c.T)
        n_c = -(-P // idx.R)
        for h in range(c.Hkv):
            mean = bf16_bits(idx.mean[b, l, h, :P])
            cent, assign, off, members = oracle.centroid_build(mean, idx.R, n_iter)
            assert np.array_equal(bf16_bits(idx.cent[b, l, h, :n_c]), cent), (b, l, h, "centroids")
            assert idx.assign[b, l, h, :P].cpu().numpy().tolist() == assign.tolist(), (b, l, h, "assignment")
            assert idx.off[b, l, h, :n_c + 1].cpu().numpy().tolist() == off.tolist(), (b, l, h, "offsets")
            assert idx.members[b, l, h, :P].cpu().numpy().tolist() == members.tolist(), (b, l, h, "members")


def check_select(wl, st, idx, l, q, M, K, cs_gpu, ps_gpu, stats, group_reduce=0, mask=None):
    """The GPU selection of every rescored unit of layer l against the oracle (see the module docstring)."""
    c = wl.cfg
    for b in range(c.B):
        P = -(-int(wl.seq_len[b]) // c.T)
        n_c = -(-P // idx.R)
        for h in range(c.Hkv):
            if mask is not None and not mask[l, h]:
                continue
            mean = bf16_bits(idx.mean[b, l, h, :P])
            cent = bf16_bits(idx.cent[b, l, h, :n_c])
            off = idx.off[b, l, h, :n_c + 1].cpu().numpy()
            mem = idx.members[b, l, h, :P].cpu().numpy()
            qg = parity.q_group(wl, q, b, h)
            ref = oracle.centroid_select(qg, mean, cent, off, mem, M, K, group_reduce)
            cnt = int(st.sel_cnt[b, l, h])
            sel = st.sel_idx[b, l, h, :cnt].cpu().numpy()
            if P == 0:
                assert cnt == 0
                continue
            # level 1: centroid scores, and the top M of the GPU's own scores against the oracle's
            cs = cs_gpu[b, h, :n_c].double().cpu().numpy()
            assert np.all(np.abs(cs - ref["cs"]) <= parity.SCORE_RTOL * max(np.abs(ref["cs"]).max(), 1e-30))
            own = oracle.topk(cs, M)
            s_m = np.sort(ref["cs"])[::-1][min(M, n_c) - 1]
            for j in set(own.tolist()) ^ set(ref["chosen"].tolist()):
                assert abs(ref["cs"][j] - s_m) <= parity.TIE_RTOL * max(abs(s_m), 1e-30), (b, h, "centroid", j)
                stats.ties += 1
            # the expanded pages: exactly the members of the GPU's top M (the pages with a score written)
            cand = sorted(p for j in own for p in mem[off[j]:off[j + 1]])
            written = np.nonzero(~torch.isnan(ps_gpu[b, h, :P]).cpu().numpy())[0].tolist()
            assert written == cand, (b, h, "expanded pages")
            # level 2: the exact top K of the GPU's candidate scores; against the oracle's over the same pages
            ps = ps_gpu[b, h, cand].double().cpu().numpy()
            assert sel.tolist() == np.array(cand)[oracle.topk(ps, K)].tolist(), (b, h, "own top K")
            ps_ref = oracle.unit_mean_scores(qg, mean[cand], len(cand), group_reduce)
            assert np.all(np.abs(ps - ps_ref) <= parity.SCORE_RTOL * max(np.abs(ps_ref).max(), 1e-30))
            want = np.array(cand)[oracle.topk(ps_ref, K)]
            s_k = np.sort(ps_ref)[::-1][min(K, len(cand)) - 1]
            for p in set(sel.tolist()) ^ set(want.tolist()):
                i = cand.index(p)
                assert abs(ps_ref[i] - s_k) <= parity.TIE_RTOL * max(abs(s_k), 1e-30), (b, h, "page", p)
                stats.ties += 1
            stats.units += 1


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("R,n_iter", [(1, 0), (4, 0), (4, 2), (8, 3), (3, 1)])
def test_build_matches_oracle(name, R, n_iter):
    cfg = CASES[name]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    idx = Index(wl, st, R)
    for l in range(cfg.L_alloc):
        idx.build(st, l, n_iter)
    torch.cuda.synchronize()
    assert st.read_err() == 0
    for l in range(cfg.L_alloc):
        check_build(wl, idx, l, n_iter)


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("group_reduce", [0, 1])
def test_two_level_selection_matches_oracle(name, group_reduce):
    cfg = CASES[name]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    R, n_iter = 4, 2
    idx = Index(wl, st, R)
    stats = parity.Stats()
    for M in (3, 10, 10 ** 6):  # few, more, every centroid
        for l in range(cfg.L_alloc):
            idx.build(st, l, n_iter)
            cs = torch.full((cfg.B, cfg.Hkv, idx.cmax), float("nan"), device="cuda")
            ps = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
            kvmm.page_score_topk_centroid(st.shape, l, wl.q[l], idx.mean, st.seq_len, R, idx.cent, idx.off,
                                          idx.members, None, M, cfg.K, st.sel_idx, st.sel_cnt, err=st.err,
                                          centroid_scores_out=cs, scores_out=ps, group_reduce=group_reduce)
            torch.cuda.synchronize()
            assert st.read_err() == 0
            check_select(wl, st, idx, l, wl.q[l], M, cfg.K, cs, ps, stats, group_reduce)
            if M >= idx.cmax:  # every centroid expanded: the flat mean-key search, up to ties
                for b in range(cfg.B):
                    P = -(-int(wl.seq_len[b]) // cfg.T)
                    for h in range(cfg.Hkv):
                        qg = parity.q_group(wl, wl.q[l], b, h)
                        s_o = oracle.unit_mean_scores(qg, bf16_bits(idx.mean[b, l, h, :P]), P, group_reduce)
                        sel = st.sel_idx[b, l, h, :int(st.sel_cnt[b, l, h])].cpu().numpy()
                        parity.check_selection(ps[b, h, :P].double().cpu().numpy(), s_o, sel, cfg.K, stats)
    print(name, group_reduce, "units", stats.units, "ties", stats.ties)


def test_rescore_mask_and_short_sequences():
    cfg = workloads.Config("short", B=3, L=2, Hq=8, Hkv=2, D=128, T=16, S=200, K=5, seed=17)
    wl = workloads.generate(cfg, device="cuda")
    wl.seq_len.copy_(torch.tensor([200, 17, 0], dtype=torch.int32))
    st = DecodeState.for_workload(wl)
    idx = Index(wl, st, 3)
    mask = torch.zeros(cfg.L, cfg.Hkv, dtype=torch.uint8, device="cuda")
    mask[0, 1] = 1
    mask[1, 0] = 1
    st.sel_idx.fill_(-5)
    st.sel_cnt.fill_(-5)
    stats = parity.Stats()
    for l in range(cfg.L):
        idx.build(st, l, 2)
        cs = torch.full((cfg.B, cfg.Hkv, idx.cmax), float("nan"), device="cuda")
        ps = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
        kvmm.page_score_topk_centroid(st.shape, l, wl.q[l], idx.mean, st.seq_len, 3, idx.cent, idx.off, idx.members,
                                      mask, 2, cfg.K, st.sel_idx, st.sel_cnt, err=st.err, centroid_scores_out=cs,
                                      scores_out=ps)
        torch.cuda.synchronize()
        assert st.read_err() == 0
        check_build(wl, idx, l, 2)
        check_select(wl, st, idx, l, wl.q[l], 2, cfg.K, cs, ps, stats, mask=mask.cpu().numpy())
    # units not rescored kept their (never written) selection
    assert int(st.sel_cnt[0, 0, 0]) == -5 and int(st.sel_cnt[2, 1, 1]) == -5
    # a rescored unit of an empty sequence selects nothing; one of a single page selects it
    assert int(st.sel_cnt[2, 0, 1]) == 0
    assert int(st.sel_cnt[1, 0, 1]) == 2 and st.sel_idx[1, 0, 1, :2].tolist() == [0, 1]


def test_identical_pages_group_under_the_first_centroid():
    cfg = workloads.Config("flat", B=1, L=1, Hq=4, Hkv=1, D=64, T=16, S=16 * 40, K=6, seed=23)
    wl = workloads.generate(cfg, device="cuda")
    wl.k_pool.copy_(wl.k_pool[:1].expand_as(wl.k_pool))  # every page the same keys
    st = DecodeState.for_workload(wl)
    idx = Index(wl, st, 4)
    idx.build(st, 0, 3)
    torch.cuda.synchronize()
    assert st.read_err() == 0
    assert torch.all(idx.assign[0, 0, 0, :40] == 0)
    assert idx.off[0, 0, 0, :11].tolist() == [0] + [40] * 10
    check_build(wl, idx, 0, 3)
