"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against an independent statement: a closed form,
a brute-force enumeration, numpy's reductions, torch's float64 softmax or
Python's set operations -- never against a retyped copy of its own formula.

Sources (FlexiCache blog summary, MLSys'26): "Core method, 2. MinMax-metadata
page scoring" (bound on the largest dot product from per-channel key min/max,
top-K pages per (layer, KV head)); "Core method, 3. Periodic reranking and
incremental promotion" (unstable heads every step, stable heads every 16
steps, promotion = current top-K minus previous top-K); "System design,
head-level block table" ([batch, layer, head, logical_block], null block).
KVDrive, "Background and key observations" (Quest: query times channel-wise
key min and max).
"""
import itertools

import numpy as np
import pytest
import torch

rng_seed = 1234


def bf16_bits_of(x: np.ndarray) -> np.ndarray:
    """Round float values to bf16 and return the bit patterns (uint16)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    u = b.astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def random_pool(rs, n_phys, T, D, scale=1.0):
    return bf16_bits_of(rs.standard_normal((n_phys, T, D)) * scale)


def to_v(vp_token_major):
    """A [n][T][D] value pool in the oracle's value layout [n][D][T]."""
    return np.ascontiguousarray(vp_token_major.transpose(0, 2, 1))


def gather_tokens(pool_f64, bt_row, T, seq_len, pages):
    rows = []
    for p in pages:
        n = min(T, seq_len - p * T)
        if n <= 0:
            continue
        rows.append(pool_f64[bt_row[p], :n, :])
    D = pool_f64.shape[-1]
    return np.concatenate(rows, axis=0) if rows else np.zeros((0, D))


# --------------------------------------------------------------------------- #
# MinMax metadata                                                             #
# --------------------------------------------------------------------------- #
def test_minmax_matches_numpy_reduction_through_permuted_table(oracle_mod):
    rs = np.random.default_rng(rng_seed)
    T, D, P = 16, 32, 9
    seq_len = 8 * T + 5  # ragged last page
    n_phys = 20
    pool = random_pool(rs, n_phys, T, D)
    bt = rs.permutation(n_phys)[:P].astype(np.int32)
    meta, err = oracle_mod.unit_minmax(pool, T, bt, seq_len)
    assert err == 0
    pf = bits_to_f64(pool)
    for p in range(P):
        rows = pf[bt[p], : min(T, seq_len - p * T)]
        assert np.array_equal(bits_to_f64(meta[p, 0]), rows.min(axis=0))
        assert np.array_equal(bits_to_f64(meta[p, 1]), rows.max(axis=0))


def test_minmax_single_token_pages_equal_the_key(oracle_mod):
    rs = np.random.default_rng(1)
    T, D, S = 1, 16, 7
    pool = random_pool(rs, S, T, D)
    bt = np.arange(S, dtype=np.int32)
    meta, err = oracle_mod.unit_minmax(pool, T, bt, S)
    assert err == 0
    assert np.array_equal(meta[:, 0, :], pool[:, 0, :])
    assert np.array_equal(meta[:, 1, :], pool[:, 0, :])


def test_minmax_signed_zero_and_invalid_rows(oracle_mod):
    T, D = 4, 2
    vals = np.array([[[0.0, 1.0], [-0.0, -1.0], [1e30, -1e30], [1e30, -1e30]]], dtype=np.float32)
    pool = bf16_bits_of(vals)
    pool[0, 0, 0] = 0x0000  # +0
    pool[0, 1, 0] = 0x8000  # -0
    meta, err = oracle_mod.unit_minmax(pool, T, np.array([0], np.int32), seq_len=2)
    assert err == 0
    # -0 orders before +0; rows 2..3 are past seq_len and must not count
    assert meta[0, 0, 0] == 0x8000 and meta[0, 1, 0] == 0x0000
    assert bits_to_f64(meta[0, 0, 1:2])[0] == -1.0 and bits_to_f64(meta[0, 1, 1:2])[0] == 1.0


def test_minmax_null_and_out_of_range_entries(oracle_mod):
    rs = np.random.default_rng(2)
    T, D = 4, 8
    pool = random_pool(rs, 3, T, D)
    bt = np.array([0, -1, 7], np.int32)
    meta, err = oracle_mod.unit_minmax(pool, T, bt, seq_len=3 * T)
    assert err == oracle_mod.ERR_NULL_BLOCK | oracle_mod.ERR_OUT_OF_RANGE
    assert not meta[1].any() and not meta[2].any()


# --------------------------------------------------------------------------- #
# Page score                                                                  #
# --------------------------------------------------------------------------- #
def test_score_hand_worked_examples(oracle_mod):
    # one head: q=(1,-2,0.5), box min=(-1,0,2), max=(3,1,4):
    #   max(-1,3) + max(0,-2) + max(1,2) = 3 + 0 + 2 = 5
    # second head q=(-1,1,-1): max(1,-3) + max(0,1) + max(-2,-4) = 1 + 1 - 2 = 0
    q = bf16_bits_of(np.array([[1, -2, 0.5], [-1, 1, -1]]))
    meta = bf16_bits_of(np.array([[[-1, 0, 2], [3, 1, 4]]]))
    assert oracle_mod.unit_scores(q[:1], meta, 1)[0] == 5.0
    assert oracle_mod.unit_scores(q[1:], meta, 1)[0] == 0.0
    assert oracle_mod.unit_scores(q, meta, 1, group_reduce=0)[0] == 5.0
    assert oracle_mod.unit_scores(q, meta, 1, group_reduce=1)[0] == 5.0
    # all-negative query on a positive box picks the minimum: -(2*1 + 3*2) = -8
    q2 = bf16_bits_of(np.array([[-2, -3]]))
    meta2 = bf16_bits_of(np.array([[[1, 2], [5, 9]]]))
    assert oracle_mod.unit_scores(q2, meta2, 1)[0] == -8.0


def test_score_is_the_maximum_over_the_box_corners(oracle_mod):
    """sum_d max(q_d min_d, q_d max_d) = max over the 2^D corners c of q.c (linear max over a box)."""
    rs = np.random.default_rng(3)
    D, G, P = 7, 3, 5
    for trial in range(20):
        q = bf16_bits_of(rs.standard_normal((G, D)) * 2)
        lo = rs.standard_normal((P, D))
        hi = lo + np.abs(rs.standard_normal((P, D)))
        meta = np.stack([bf16_bits_of(lo), bf16_bits_of(hi)], axis=1)
        s = oracle_mod.unit_scores(q, meta, P, group_reduce=0)
        smax = oracle_mod.unit_scores(q, meta, P, group_reduce=1)
        qf = bits_to_f64(q)
        mf = bits_to_f64(meta)
        for p in range(P):
            per_head = []
            for g in range(G):
                best = max(sum(qf[g, d] * mf[p, c[d], d] for d in range(D))
                           for c in itertools.product((0, 1), repeat=D))
                per_head.append(best)
            assert s[p] == pytest.approx(sum(per_head), rel=1e-12, abs=1e-12)
            assert smax[p] == pytest.approx(max(per_head), rel=1e-12, abs=1e-12)


def test_score_bounds_every_true_dot_product(oracle_mod):
    rs = np.random.default_rng(4)
    T, D, G, P = 16, 64, 4, 12
    pool = random_pool(rs, P, T, D)
    pool[:, :, :4] = bf16_bits_of(bits_to_f64(pool[:, :, :4]) * 8)  # outlier channels
    bt = np.arange(P, dtype=np.int32)
    seq_len = P * T - 3
    meta, _ = oracle_mod.unit_minmax(pool, T, bt, seq_len)
    q = bf16_bits_of(rs.standard_normal((G, D)))
    qf, kf = bits_to_f64(q), bits_to_f64(pool)
    s_sum = oracle_mod.unit_scores(q, meta, P, 0)
    for g in range(G):
        s_g = oracle_mod.unit_scores(q[g:g + 1], meta, P, 0)
        for p in range(P):
            n = min(T, seq_len - p * T)
            dots = kf[p, :n] @ qf[g]
            assert s_g[p] >= dots.max() - 1e-9
    for p in range(P):
        n = min(T, seq_len - p * T)
        assert s_sum[p] >= (kf[p, :n] @ qf.sum(axis=0)).max() - 1e-9


def test_score_single_token_pages_equal_the_dot_product(oracle_mod):
    rs = np.random.default_rng(5)
    D, P = 32, 10
    pool = random_pool(rs, P, 1, D)
    meta, _ = oracle_mod.unit_minmax(pool, 1, np.arange(P, dtype=np.int32), P)
    q = bf16_bits_of(rs.standard_normal((1, D)))
    s = oracle_mod.unit_scores(q, meta, P)
    ref = bits_to_f64(pool)[:, 0, :] @ bits_to_f64(q)[0]
    assert np.allclose(s, ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- #
# Top-K                                                                       #
# --------------------------------------------------------------------------- #
def test_topk_matches_brute_force_sort_with_ties(oracle_mod):
    rs = np.random.default_rng(6)
    for trial in range(300):
        P = int(rs.integers(1, 17))
        K = int(rs.integers(1, P + 3))
        scores = rs.integers(-3, 4, size=P).astype(np.float64)  # many exact ties
        want = sorted(sorted(range(P), key=lambda p: (-scores[p], p))[:min(K, P)])
        got = oracle_mod.topk(scores, K)
        assert got.tolist() == want


def test_topk_takes_all_pages_when_budget_covers_them(oracle_mod):
    s = np.array([0.5, -1.0, 3.0])
    assert oracle_mod.topk(s, 3).tolist() == [0, 1, 2]
    assert oracle_mod.topk(s, 10).tolist() == [0, 1, 2]
    assert oracle_mod.topk(s, 1).tolist() == [2]


# --------------------------------------------------------------------------- #
# Promotion diff                                                              #
# --------------------------------------------------------------------------- #
def test_set_difference_matches_python_sets(oracle_mod):
    rs = np.random.default_rng(7)
    cases = [([], []), ([1, 2, 3], [1, 2, 3]), ([1, 2], [3, 4]), ([], [5]), ([5], [])]
    for _ in range(200):
        a = sorted(rs.choice(40, size=int(rs.integers(0, 20)), replace=False).tolist())
        b = sorted(rs.choice(40, size=int(rs.integers(0, 20)), replace=False).tolist())
        cases.append((a, b))
    for a, b in cases:
        assert oracle_mod.set_difference(a, b).tolist() == sorted(set(a) - set(b))
        assert oracle_mod.set_difference(b, a).tolist() == sorted(set(b) - set(a))


def test_rerank_schedule(oracle_mod):
    assert all(oracle_mod.rescored(True, s) for s in range(40))
    assert [s for s in range(40) if oracle_mod.rescored(False, s)] == [0, 16, 32]


# --------------------------------------------------------------------------- #
# Attention                                                                   #
# --------------------------------------------------------------------------- #
def torch_attention(q_bits, k_rows, v_rows, scale):
    q = torch.tensor(bits_to_f64(q_bits))
    k = torch.tensor(k_rows)
    v = torch.tensor(v_rows)
    z = (q @ k.T) * scale
    return (torch.softmax(z, dim=-1) @ v).numpy(), torch.logsumexp(z, dim=-1).numpy()


def test_sparse_attention_matches_torch_softmax(oracle_mod):
    rs = np.random.default_rng(8)
    T, D, G, P = 16, 64, 4, 10
    n_phys = 16
    seq_len = P * T - 7
    kp, vp = random_pool(rs, n_phys, T, D), random_pool(rs, n_phys, T, D)
    bt = rs.permutation(n_phys)[:P].astype(np.int32)
    q = bf16_bits_of(rs.standard_normal((G, D)))
    sel = np.array([0, 3, 4, 9], np.int32)  # includes the ragged last page
    out, lse, err = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, bt, seq_len, sel)
    assert err == 0
    kr = gather_tokens(bits_to_f64(kp), bt, T, seq_len, sel)
    vr = gather_tokens(bits_to_f64(vp), bt, T, seq_len, sel)
    ref, ref_lse = torch_attention(q, kr, vr, D ** -0.5)
    assert np.allclose(out, ref, rtol=0, atol=1e-12)
    assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_all_pages_selected_equals_dense_attention(oracle_mod):
    rs = np.random.default_rng(9)
    T, D, G, P = 16, 64, 4, 64  # the tiny shape: 1024 tokens, all 64 pages selected
    kp, vp = random_pool(rs, P, T, D), random_pool(rs, P, T, D)
    bt = np.arange(P, dtype=np.int32)
    q = bf16_bits_of(rs.standard_normal((G, D)))
    sparse, lse_s, _ = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, bt, P * T, np.arange(P))
    dense, lse_d, _ = oracle_mod.unit_dense_attention(q, kp, to_v(vp), T, bt, P * T)
    assert np.array_equal(sparse, dense) and np.array_equal(lse_s, lse_d)
    ref, ref_lse = torch_attention(q, bits_to_f64(kp).reshape(-1, D), bits_to_f64(vp).reshape(-1, D), D ** -0.5)
    assert np.allclose(dense, ref, rtol=0, atol=1e-12)
    assert np.allclose(lse_d, ref_lse, rtol=0, atol=1e-12)


def test_single_token_gives_its_value_and_equal_keys_give_the_mean(oracle_mod):
    rs = np.random.default_rng(10)
    T, D, G = 16, 32, 2
    kp, vp = random_pool(rs, 2, T, D), random_pool(rs, 2, T, D)
    q = bf16_bits_of(rs.standard_normal((G, D)))
    out, lse, _ = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, np.array([0], np.int32), 1, [0])
    assert np.array_equal(out, np.repeat(bits_to_f64(vp[0, :1]), G, axis=0))
    assert np.allclose(lse, bits_to_f64(q) @ bits_to_f64(kp[0, 0]) * D ** -0.5, atol=1e-12)
    kp[1] = kp[1, 0]  # every key of page 1 identical -> uniform weights
    out, _, _ = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, np.array([1], np.int32), T, [0])
    assert np.allclose(out, np.repeat(bits_to_f64(vp[1]).mean(axis=0)[None], G, axis=0), atol=1e-12)


def test_empty_selection_gives_zero_output(oracle_mod):
    rs = np.random.default_rng(11)
    kp, vp = random_pool(rs, 1, 4, 8), random_pool(rs, 1, 4, 8)
    q = bf16_bits_of(rs.standard_normal((2, 8)))
    out, lse, err = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), 4, np.array([0], np.int32), 4, [])
    assert err == 0 and not out.any() and np.all(np.isneginf(lse))


def test_permuted_pool_is_transparent_and_null_block_is_skipped(oracle_mod):
    rs = np.random.default_rng(12)
    T, D, G, P = 16, 32, 4, 8
    kp, vp = random_pool(rs, P, T, D), random_pool(rs, P, T, D)
    q = bf16_bits_of(rs.standard_normal((G, D)))
    ident = np.arange(P, dtype=np.int32)
    perm = rs.permutation(P).astype(np.int32)
    kperm, vperm = np.empty_like(kp), np.empty_like(vp)
    kperm[perm], vperm[perm] = kp, vp  # logical page p lives at physical perm[p]
    sel = [1, 2, 6]
    a, la, _ = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, ident, P * T, sel)
    b, lb, _ = oracle_mod.unit_sparse_attention(q, kperm, to_v(vperm), T, perm, P * T, sel)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    # a null entry on an unselected page changes nothing
    bt_null = ident.copy()
    bt_null[4] = -1
    c, _, err = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, bt_null, P * T, sel)
    assert err == 0 and np.array_equal(a, c)
    # a selected null page is reported and contributes nothing
    bt_null[2] = -1
    d, _, err = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, bt_null, P * T, sel)
    e, _, _ = oracle_mod.unit_sparse_attention(q, kp, to_v(vp), T, ident, P * T, [1, 6])
    assert err == oracle_mod.ERR_NULL_BLOCK and np.array_equal(d, e)


# --------------------------------------------------------------------------- #
# One decode step of a unit (append, rerank schedule, diff, attention)        #
# --------------------------------------------------------------------------- #
def test_unit_step_follows_the_rerank_schedule(oracle_mod):
    rs = np.random.default_rng(13)
    T, D, G, K = 16, 32, 4, 3
    S0, steps = 5 * T - 2, 6
    Pmax = -(-(S0 + steps) // T)
    kp, vp = random_pool(rs, Pmax, T, D), to_v(random_pool(rs, Pmax, T, D))
    bt = np.arange(Pmax, dtype=np.int32)
    meta, _ = oracle_mod.unit_minmax(kp, T, bt, S0)
    st = oracle_mod.UnitState(kp, vp, T, bt, meta, K)
    prev = []
    for step in range(steps):
        seq = S0 + 1 + step
        nk = bf16_bits_of(rs.standard_normal((1, D)) * 3)
        nv = bf16_bits_of(rs.standard_normal((1, D)))
        q = bf16_bits_of(rs.standard_normal((G, D)))
        resc = oracle_mod.rescored(False, step, period=3)
        out, lse, err = oracle_mod.unit_step(st, seq, nk, nv, q, resc)
        assert err == 0
        # the new token landed and the metadata of its page covers it
        assert np.array_equal(st.k_pool[(seq - 1) // T, (seq - 1) % T], nk[0])
        assert np.array_equal(st.v_pool[(seq - 1) // T, :, (seq - 1) % T], nv[0])
        full_meta, _ = oracle_mod.unit_minmax(st.k_pool, T, bt, seq)
        P = -(-seq // T)
        assert np.array_equal(st.meta[:P], full_meta[:P])
        cur = st.sel[: st.sel_cnt[0]].tolist()
        if resc:
            scores = oracle_mod.unit_scores(q, st.meta, P)
            want = sorted(sorted(range(P), key=lambda p: (-scores[p], p))[:K])
            assert cur == want
            assert st.promoted[: st.n_promoted[0]].tolist() == sorted(set(cur) - set(prev))
            assert st.evicted[: st.n_evicted[0]].tolist() == sorted(set(prev) - set(cur))
        else:
            assert cur == prev and st.n_promoted[0] == 0
        ref, _, _ = oracle_mod.unit_sparse_attention(q, st.k_pool, st.v_pool, T, bt, seq, cur)
        assert np.array_equal(out, ref)
        prev = cur
