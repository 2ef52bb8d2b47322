"""GPU parity of promote_pages: promoted pages from pinned host memory into recycled blocks.

FlexiCache blog summary (MLSys'26), "Core method, 3" (only the promoted pages
move), "Core method, 4" (a UVA kernel reads the pinned host KV directly, with
a bounded grid) and "System design, head-level block table" (evicted pages'
blocks are reused; evicted entries point at the null block).  The kernel must
leave exactly the oracle's table, pools, moved and freed lists, for several
grid bounds and a partial rescore mask; attention over the new selection then
equals the oracle's attention over the host store.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_minmax_gb300 import kvmm
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


def setup(B, L, Hkv, D, T, Pmax, K, seed, grow=0, shrink=0):
    """Host store (pinned), pools holding each unit's previous selection, the new selections' diff lists."""
    rng = np.random.default_rng(seed)
    units = B * L * Hkv
    host_k = torch.randn(B, L, Hkv, Pmax, T, D, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    host_v = torch.randn(B, L, Hkv, Pmax, D, T, dtype=torch.float32).to(torch.bfloat16).pin_memory()
    n_phys = units * K + 8
    k_pool = torch.zeros(n_phys, T, D, dtype=torch.bfloat16)
    v_pool = torch.zeros(n_phys, D, T, dtype=torch.bfloat16)
    bt = np.full((B, L, Hkv, Pmax), -1, dtype=np.int32)
    prom = np.zeros((B, L, Hkv, K), dtype=np.int32)
    evic = np.zeros((B, L, Hkv, K), dtype=np.int32)
    pcnt = np.zeros((B, L, Hkv), dtype=np.int32)
    ecnt = np.zeros((B, L, Hkv), dtype=np.int32)
    blocks = rng.permutation(n_phys)
    nb = 0
    cur_sel = {}
    for b in range(B):
        for l in range(L):
            for h in range(Hkv):
                prev = np.sort(rng.choice(Pmax, K, replace=False))
                for pg in prev:
                    blk = int(blocks[nb])
                    nb += 1
                    bt[b, l, h, pg] = blk
                    k_pool[blk] = host_k[b, l, h, pg]
                    v_pool[blk] = host_v[b, l, h, pg]
                keep = prev[rng.random(len(prev)) < 0.65]
                rest = np.setdiff1d(np.arange(Pmax), prev)
                new = rng.choice(rest, max(0, K + grow - shrink - len(keep)), replace=False)
                cur = np.sort(np.concatenate([keep, new])).astype(np.int32)
                cur_sel[(b, l, h)] = cur
                p_ = np.array(sorted(set(cur) - set(prev)), dtype=np.int32)[:K]
                e_ = np.array(sorted(set(prev) - set(cur)), dtype=np.int32)[:K]
                prom[b, l, h, :len(p_)] = p_
                evic[b, l, h, :len(e_)] = e_
                pcnt[b, l, h] = len(p_)
                ecnt[b, l, h] = len(e_)
    return dict(host_k=host_k, host_v=host_v, k_pool=k_pool, v_pool=v_pool, bt=bt, prom=prom, evic=evic, pcnt=pcnt,
                ecnt=ecnt, n_phys=n_phys, cur=cur_sel)


def run_oracle(st, layer, mask, B, Hkv, T):
    bt = st["bt"].copy()
    kp = bf16_bits(st["k_pool"]).reshape(st["n_phys"], -1).copy()
    vp = bf16_bits(st["v_pool"]).reshape(st["n_phys"], -1).copy()
    hk, hv = bf16_bits(st["host_k"]), bf16_bits(st["host_v"])
    moved, freed = {}, {}
    err = 0
    for b in range(B):
        for h in range(Hkv):
            if mask is not None and not mask[layer, h]:
                continue
            row = bt[b, layer, h]
            e, m, f = oracle.unit_promote(row, st["n_phys"], st["prom"][b, layer, h, :st["pcnt"][b, layer, h]],
                                          st["evic"][b, layer, h, :st["ecnt"][b, layer, h]],
                                          hk[b, layer, h].reshape(hk.shape[3], -1), hv[b, layer, h].reshape(hv.shape[3], -1),
                                          kp, vp, T)
            err |= e
            moved[(b, h)] = m
            freed[(b, h)] = f
    return bt, kp, vp, moved, freed, err


@pytest.mark.parametrize("D,T,max_ctas,grow,shrink,masked", [
    (64, 16, 0, 0, 0, False), (128, 16, 1, 0, 0, True), (128, 32, 4, 2, 0, False), (64, 32, 3, 0, 3, True)])
def test_promotion_matches_the_oracle(D, T, max_ctas, grow, shrink, masked):
    B, L, Hkv, Pmax, K = 2, 2, 4, 48, 12
    st = setup(B, L, Hkv, D, T, Pmax, K, seed=D + T + max_ctas, grow=grow, shrink=shrink)
    shape = kvmm.make_shape(B, L, Hkv * 2, Hkv, D, T, Pmax, K, st["n_phys"])
    mask = None
    if masked:
        mask = np.zeros((L, Hkv), dtype=np.uint8)
        mask[:, 1::2] = 1
    dev = lambda a: torch.tensor(a, device="cuda")
    k_pool, v_pool = st["k_pool"].cuda(), st["v_pool"].cuda()
    bt = dev(st["bt"])
    moved = torch.full((B, L, Hkv), -9, dtype=torch.int32, device="cuda")
    freed = torch.full((B, L, Hkv, K), -9, dtype=torch.int32, device="cuda")
    freed_cnt = torch.full((B, L, Hkv), -9, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for layer in range(L):
        kvmm.promote_pages(shape, layer, dev(mask) if mask is not None else None, dev(st["prom"]), dev(st["pcnt"]),
                           dev(st["evic"]), dev(st["ecnt"]), st["host_k"], st["host_v"], k_pool, v_pool, bt,
                           moved=moved, freed=freed, freed_cnt=freed_cnt, max_ctas=max_ctas, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want_bt = st["bt"].copy()
    want_kp = bf16_bits(st["k_pool"]).reshape(st["n_phys"], -1).copy()
    want_vp = bf16_bits(st["v_pool"]).reshape(st["n_phys"], -1).copy()
    for layer in range(L):
        st["bt"] = want_bt
        st["k_pool"] = torch.tensor(want_kp.view(np.int16)).view(torch.bfloat16).reshape(st["n_phys"], T, D)
        st["v_pool"] = torch.tensor(want_vp.view(np.int16)).view(torch.bfloat16).reshape(st["n_phys"], D, T)
        want_bt, want_kp, want_vp, w_moved, w_freed, w_err = run_oracle(st, layer, mask, B, Hkv, T)
        assert w_err == 0
        for (b, h), mv in w_moved.items():
            assert int(moved[b, layer, h]) == mv
            fc = int(freed_cnt[b, layer, h])
            assert fc == len(w_freed[(b, h)])
            assert freed[b, layer, h, :fc].cpu().tolist() == w_freed[(b, h)].tolist()
    np.testing.assert_array_equal(bt.cpu().numpy(), want_bt)
    np.testing.assert_array_equal(bf16_bits(k_pool).reshape(st["n_phys"], -1), want_kp)
    np.testing.assert_array_equal(bf16_bits(v_pool).reshape(st["n_phys"], -1), want_vp)


def test_attention_after_promotion_reads_the_host_pages():
    B, L, Hkv, D, T, Pmax, K, G = 2, 1, 4, 128, 16, 64, 16, 4
    st = setup(B, L, Hkv, D, T, Pmax, K, seed=11)
    shape = kvmm.make_shape(B, L, Hkv * G, Hkv, D, T, Pmax, K, st["n_phys"])
    dev = lambda a: torch.tensor(a, device="cuda")
    k_pool, v_pool, bt = st["k_pool"].cuda(), st["v_pool"].cuda(), dev(st["bt"])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvmm.promote_pages(shape, 0, None, dev(st["prom"]), dev(st["pcnt"]), dev(st["evic"]), dev(st["ecnt"]),
                       st["host_k"], st["host_v"], k_pool, v_pool, bt, err=err)
    sel = np.zeros((B, L, Hkv, K), dtype=np.int32)
    cnt = np.zeros((B, L, Hkv), dtype=np.int32)
    for (b, l, h), cur in st["cur"].items():
        sel[b, l, h, :len(cur)] = cur
        cnt[b, l, h] = len(cur)
    seq = torch.full((B,), Pmax * T - 3, dtype=torch.int32, device="cuda")
    q = torch.randn(B, Hkv * G, D, device="cuda").to(torch.bfloat16)
    out = torch.zeros(B, Hkv * G, D, device="cuda")
    lse = torch.zeros(B, Hkv * G, device="cuda")
    kvmm.sparse_paged_decode_attn(shape, 0, q, k_pool, v_pool, bt, seq, dev(sel), dev(cnt), out, None, lse=lse, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    hk, hv = bf16_bits(st["host_k"]), bf16_bits(st["host_v"])
    qb = bf16_bits(q)
    ident = np.arange(Pmax, dtype=np.int32)
    for b in range(B):
        for h in range(Hkv):
            cur = st["cur"][(b, 0, h)]
            o, _, e = oracle.unit_sparse_attention(qb[b, h * G:(h + 1) * G], hk[b, 0, h].reshape(-1),
                                                   hv[b, 0, h].reshape(-1), T, ident, Pmax * T - 3, cur)
            assert e == 0
            d = np.abs(out[b, h * G:(h + 1) * G].cpu().numpy() - o)
            assert d.max() <= 2e-3 and d.sum() / np.abs(o).sum() <= 1e-3
