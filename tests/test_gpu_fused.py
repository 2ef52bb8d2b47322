"""GPU parity of page_score_topk_attn (scoring, then attention that selects its
own pages) against the CPU oracle and against the two separate calls.

The fused call must select exactly what page_score_topk selects (bit-exact
scores, indices and counts) and attend within the attention tolerance of the
oracle; repeated launches on one workspace, partial rescore masks, ragged
and empty units, null blocks, both group reductions, every (D, T)
instantiation and the long-table route each have a case.
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
    "permuted": scaled(CONFIGS[3], B=2, L=1, S=8192 + 5, K=64, n_planted=32),
    "gqa5-t32": scaled(CONFIGS[5], B=2, L=2, S=4096 - 7, K=16, n_planted=8, ragged=True, layers_alloc=None),
    "d64-g8": workloads.Config("d64-g8", B=2, L=1, Hq=16, Hkv=2, D=64, T=16, S=1500, K=12, key_dist="chanscale",
                               n_planted=6, ragged=True, permuted_pool=True, seed=77),
    "g1-d128-t32": workloads.Config("g1-d128", B=1, L=1, Hq=4, Hkv=4, D=128, T=32, S=777, K=5, seed=78),
    "d64-t32": workloads.Config("d64-t32", B=3, L=1, Hq=8, Hkv=2, D=64, T=32, S=3000, K=40, ragged=True, seed=79),
    "big-k": scaled(CONFIGS[2], B=1, L=1, S=32768, K=1000, n_planted=64),
    "p3000": scaled(CONFIGS[2], B=1, L=1, S=3000 * 16 - 9, K=200, n_planted=32, ragged=True),
    # 32768 pages: the selection does not fit the attention CTA; the call runs the separate kernels
    "p32768": scaled(CONFIGS[2], B=1, L=1, S=32768 * 16, K=300, n_planted=32),
}


def fused_states(cfg, group_reduce=0):
    wl = workloads.generate(cfg, device="cuda")
    fused = DecodeState.for_workload(wl, group_reduce=group_reduce)
    sep = DecodeState.for_workload(wl, group_reduce=group_reduce)
    fused.build_metadata()
    sep.meta.copy_(fused.meta)
    return wl, fused, sep


def run_layer(wl, fused, sep, l, q, mask=None):
    cfg = wl.cfg
    sf = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    ss = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    fused.select_attend(l, q, rescore_mask=mask, scores_out=sf)
    sep.select(l, q, rescore_mask=mask, scores_out=ss)
    sep.attend(l, q)
    torch.cuda.synchronize()
    return sf, ss


def assert_same_selection(fused, sep, sf=None, ss=None):
    assert torch.equal(fused.sel_cnt, sep.sel_cnt)
    for idx in torch.nonzero(torch.ones_like(fused.sel_cnt)).tolist():
        n = int(fused.sel_cnt[tuple(idx)])
        assert torch.equal(fused.sel_idx[tuple(idx)][:n], sep.sel_idx[tuple(idx)][:n]), idx
    if sf is not None:
        assert torch.equal(torch.nan_to_num(sf, nan=7.0), torch.nan_to_num(ss, nan=7.0)), "scores differ"


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_matches_oracle_and_separate_calls(name):
    cfg = CASES[name]
    wl, fused, sep = fused_states(cfg)
    full = (parity.bf16_bits(wl.k_pool), parity.bf16_bits(wl.v_pool)) if wl.n_phys * cfg.T * cfg.D <= (1 << 24) else None
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        sf, ss = run_layer(wl, fused, sep, l, wl.q[l])
        assert fused.read_err() == 0 and sep.read_err() == 0
        assert_same_selection(fused, sep, sf, ss)
        for b in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wl, fused, l, b, h, wl.q[l], sf, stats, full=full)
        d = (fused.out[l] - sep.out[l]).abs().max().item()
        assert d <= 2e-5, f"fused vs separate attention differ by {d}"
    stats.check()
    print(name, "units", stats.units, "ties", stats.ties, "max-abs", stats.max_abs)


def test_repeated_launches_on_one_workspace():
    """Consecutive launches with changing queries on one workspace: every launch leaves what the separate
    calls leave."""
    cfg = CASES["llama-ragged"]
    wl, fused, sep = fused_states(cfg)
    qs = workloads.drift_queries(wl, 6)
    for step in range(6):
        q = qs[step]
        for l in range(cfg.L):
            sf, ss = run_layer(wl, fused, sep, l, q[l])
            assert fused.read_err() == 0
            assert_same_selection(fused, sep, sf, ss)
            assert (fused.out[l] - sep.out[l]).abs().max().item() <= 2e-5


def test_partial_rescore_mask_keeps_stable_selections():
    cfg = CASES["llama-ragged"]
    wl, fused, sep = fused_states(cfg)
    for l in range(cfg.L):
        run_layer(wl, fused, sep, l, wl.q[l])
    mask = torch.zeros(cfg.L_alloc, cfg.Hkv, dtype=torch.uint8, device="cuda")
    mask[:, 1::3] = 1
    before = fused.sel_idx.clone()
    q2 = torch.roll(wl.q, 1, dims=2)  # new queries: rescored units change their selection
    for l in range(cfg.L):
        sf, ss = run_layer(wl, fused, sep, l, q2[l], mask=mask)
        assert fused.read_err() == 0
        assert_same_selection(fused, sep, sf, ss)
        assert (fused.out[l] - sep.out[l]).abs().max().item() <= 2e-5
    keep = mask[: cfg.L].cpu() == 0
    for l in range(cfg.L):
        for h in range(cfg.Hkv):
            if keep[l, h]:
                assert torch.equal(fused.sel_idx[:, l, h], before[:, l, h])


def test_group_max_mode():
    cfg = CASES["gqa5-t32"]
    wl, fused, sep = fused_states(cfg, group_reduce=1)
    stats = parity.Stats()
    for l in range(cfg.L_alloc):
        sf, ss = run_layer(wl, fused, sep, l, wl.q[l])
        assert fused.read_err() == 0
        assert_same_selection(fused, sep, sf, ss)
        for b in range(cfg.B):
            for h in range(cfg.Hkv):
                parity.check_unit(wl, fused, l, b, h, wl.q[l], sf, stats, group_reduce=1)
    stats.check()


def test_short_and_empty_units():
    cfg = workloads.Config("short", B=3, L=1, Hq=8, Hkv=2, D=128, T=16, S=40, K=8, seed=5)
    wl = workloads.generate(cfg, device="cuda")
    wl.seq_len.copy_(torch.tensor([40, 1, 0], dtype=torch.int32))
    fused = DecodeState.for_workload(wl)
    fused.build_metadata()
    sf = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    fused.select_attend(0, wl.q[0], scores_out=sf)
    torch.cuda.synchronize()
    assert fused.read_err() == 0
    assert fused.sel_cnt[:, 0].tolist() == [[3, 3], [1, 1], [0, 0]]
    stats = parity.Stats()
    for b in range(2):
        for h in range(2):
            parity.check_unit(wl, fused, 0, b, h, wl.q[0], sf, stats)
    stats.check()
    assert torch.all(fused.out[0, 2] == 0)
    assert torch.all(torch.isneginf(fused.lse[0, 2]))


def test_null_blocks_outside_the_selection_are_never_read():
    cfg = CASES["llama-ragged"]
    wl, fused, sep = fused_states(cfg)
    for l in range(cfg.L):
        fused.select_attend(l, wl.q[l])
    torch.cuda.synchronize()
    ref = fused.out.clone()
    sel_mask = torch.zeros(cfg.B, cfg.L, cfg.Hkv, cfg.Pmax, dtype=torch.bool, device="cuda")
    for b in range(cfg.B):
        for l in range(cfg.L):
            for h in range(cfg.Hkv):
                n = int(fused.sel_cnt[b, l, h])
                sel_mask[b, l, h, fused.sel_idx[b, l, h, :n].long()] = True
    wl.block_table.masked_fill_(~sel_mask, kvmm.NULL_BLOCK)
    for l in range(cfg.L):
        fused.select_attend(l, wl.q[l])
    torch.cuda.synchronize()
    assert fused.read_err() == 0
    assert torch.equal(fused.out, ref)
    # a selected page mapped to the null block is reported and skipped
    victim = int(fused.sel_idx[0, 0, 0, 3])
    wl.block_table[0, 0, 0, victim] = kvmm.NULL_BLOCK
    fused.select_attend(0, wl.q[0])
    torch.cuda.synchronize()
    assert fused.read_err() & kvmm.ERR_NULL_BLOCK
    assert not fused.read_err() & kvmm.ERR_TIMEOUT
    stats = parity.Stats()
    parity.check_unit(wl, fused, 0, 0, 0, wl.q[0], None, stats, check_meta=False)
    stats.check()


def test_small_workspace_is_rejected():
    cfg = CASES["tiny"]
    wl, fused, _ = fused_states(cfg)
    small = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvmm.KvmmError) as e:
        kvmm.page_score_topk_attn(fused.shape, 0, wl.q[0], fused.meta, wl.k_pool, wl.v_pool, wl.block_table,
                                  wl.seq_len, None, cfg.K, fused.sel_idx, fused.sel_cnt, fused.out[0], small)
    assert e.value.status == kvmm.WORKSPACE_TOO_SMALL
