"""GPU parity of the mean-key scorer (kv_meankey_update, page_score_topk_mean).

KVDrive, "Method details": each page's mean key is its representative.  The
metadata must equal the oracle's bit for bit (the rounding is taken in the
kernel's fp32 precision on both sides), after a full build and after an
append; scores must match within 1e-5 relative; selections follow the same
tie rules as the MinMax path.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm, workloads
from paged_kv_cache_minmax_gb300.runtime import DecodeState
from paged_kv_cache_minmax_gb300.workloads import bf16_bits

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
    "d128-t16": workloads.Config("mk1", B=2, L=2, Hq=16, Hkv=4, D=128, T=16, S=3000, K=24, key_dist="outlier",
                                 n_planted=12, ragged=True, seed=31),
    "d64-t32-g5": workloads.Config("mk2", B=2, L=1, Hq=20, Hkv=4, D=64, T=32, S=2500, K=16, key_dist="chanscale",
                                   n_planted=8, permuted_pool=True, seed=32),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("group_reduce", [0, 1])
def test_mean_metadata_scores_and_selection(name, group_reduce):
    cfg = CASES[name]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl, group_reduce=group_reduce)
    shape = st.shape
    mean = torch.zeros(cfg.B, cfg.L_alloc, cfg.Hkv, cfg.Pmax, cfg.D, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scores = torch.full((cfg.B, cfg.Hkv, cfg.Pmax), float("nan"), device="cuda")
    kp = bf16_bits(wl.k_pool).reshape(-1, cfg.T, cfg.D)
    for l in range(cfg.L_alloc):
        kvmm.kv_meankey_update(shape, l, None, wl.seq_len, wl.k_pool, wl.block_table, mean, err=err)
        kvmm.page_score_topk_mean(shape, l, wl.q[l], mean, wl.seq_len, None, cfg.K, st.sel_idx, st.sel_cnt,
                                  st.workspace, err=err, scores_out=scores, group_reduce=group_reduce)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        mb = bf16_bits(mean)
        for b in range(cfg.B):
            seq = int(wl.seq_len[b])
            P = -(-seq // cfg.T)
            for h in range(cfg.Hkv):
                row = wl.block_table[b, l, h].cpu().numpy()
                want, e = oracle.unit_meankey(kp, cfg.T, row, seq)
                assert e == 0
                assert np.array_equal(mb[b, l, h, :P], want[:P]), (b, l, h)
                qg = bf16_bits(wl.q[l, b, h * cfg.G:(h + 1) * cfg.G])
                s_o = oracle.unit_mean_scores(qg, want, P, group_reduce)
                s_g = scores[b, h, :P].double().cpu().numpy()
                assert np.abs(s_g - s_o).max() <= 1e-5 * max(np.abs(s_o).max(), 1e-30)
                sel = st.sel_idx[b, l, h, :int(st.sel_cnt[b, l, h])].cpu().numpy()
                assert sel.tolist() == oracle.topk(s_g, cfg.K).tolist()
                kth = np.sort(s_o)[::-1][min(cfg.K, P) - 1]
                for p in set(sel.tolist()) ^ set(oracle.topk(s_o, cfg.K).tolist()):
                    assert abs(s_o[p] - kth) <= 1e-5 * abs(kth)


def test_append_refresh_equals_a_rebuild():
    cfg = CASES["d128-t16"]
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    shape = st.shape
    full = torch.zeros(cfg.B, cfg.L_alloc, cfg.Hkv, cfg.Pmax, cfg.D, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvmm.kv_meankey_update(shape, 0, None, wl.seq_len, wl.k_pool, wl.block_table, full, err=err)
    inc = full.clone()
    nk, nv = workloads.step_tokens(wl, 0)
    st.append(0, nk[0], nv[0])  # rewrites the token at seq_len - 1
    begin = (wl.seq_len - 1).to(torch.int32)
    kvmm.kv_meankey_update(shape, 0, begin, wl.seq_len, wl.k_pool, wl.block_table, inc, err=err)
    kvmm.kv_meankey_update(shape, 0, None, wl.seq_len, wl.k_pool, wl.block_table, full, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and st.read_err() == 0
    assert torch.equal(inc, full)
