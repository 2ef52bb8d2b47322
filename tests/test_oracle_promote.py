"""Pins of the oracle's page promotion (physical block reuse, null-block rewrite).

FlexiCache blog summary (MLSys'26): "Core method, 3. Periodic reranking and
incremental promotion" (only current top-K minus previous top-K moves),
"Core method, 4. Overlapping transfer and compute" (promoted pages come from
the host KV), "System design, head-level block table" (evicted pages' blocks
are reused for promoted pages; evicted entries point at the null block).

The pins do not retype the pairing rule: they check that no block is created
or lost, that every page of the new selection then holds exactly its host
page, that attention over the new selection after promotion equals attention
over the host store itself, and the surplus cases by counting.
"""
import numpy as np
import pytest


T, D = 16, 64




def bf16_bits(rng, shape):
    x = rng.standard_normal(shape).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def resident_unit(rng, Pmax, prev, spare=4):
    """A unit whose pool holds exactly the pages `prev` (from its host store), in shuffled blocks."""
    host_k = bf16_bits(rng, (Pmax, T * D))
    host_v = bf16_bits(rng, (Pmax, T * D))
    n_phys = len(prev) + spare
    blocks = rng.permutation(n_phys)[:len(prev)]
    bt = np.full(Pmax, -1, dtype=np.int32)
    k_pool = np.zeros((n_phys, T * D), dtype=np.uint16)
    v_pool = np.zeros((n_phys, T * D), dtype=np.uint16)
    for pg, blk in zip(prev, blocks):
        bt[pg] = blk
        k_pool[blk] = host_k[pg]
        v_pool[blk] = host_v[pg]
    return host_k, host_v, bt, k_pool, v_pool, n_phys


def diff_lists(prev, cur):
    return np.array(sorted(set(cur) - set(prev)), dtype=np.int32), np.array(sorted(set(prev) - set(cur)), dtype=np.int32)


def test_blocks_are_reused_not_created_or_lost_and_pages_land_in_them(oracle_mod):
    rng = np.random.default_rng(5)
    prev, cur = [1, 3, 5, 7, 11], [1, 4, 7, 9, 11]
    hk, hv, bt, kp, vp, n_phys = resident_unit(rng, 16, prev)
    before = sorted(bt[bt >= 0].tolist())
    promoted, evicted = diff_lists(prev, cur)
    err, moved, freed = oracle_mod.unit_promote(bt, n_phys, promoted, evicted, hk, hv, kp, vp, T)
    assert err == 0 and moved == 2 and len(freed) == 0
    assert sorted(bt[bt >= 0].tolist()) == before  # the same blocks, reassigned
    assert set(np.nonzero(bt >= 0)[0].tolist()) == set(cur)
    for pg in cur:
        assert np.array_equal(kp[bt[pg]], hk[pg]) and np.array_equal(vp[bt[pg]], hv[pg])
    assert bt[3] == -1 and bt[5] == -1


def test_attention_after_promotion_equals_attention_over_the_host_store(oracle_mod):
    rng = np.random.default_rng(6)
    Pmax, K, G, seq = 40, 10, 4, 40 * T - 5
    prev = np.sort(rng.choice(Pmax, K, replace=False))
    keep = prev[rng.random(K) < 0.6]
    cur = np.sort(np.concatenate([keep, rng.choice(np.setdiff1d(np.arange(Pmax), prev), K - len(keep), replace=False)]))
    hk, hv, bt, kp, vp, n_phys = resident_unit(rng, Pmax, prev.tolist())
    promoted, evicted = diff_lists(prev.tolist(), cur.tolist())
    err, moved, _ = oracle_mod.unit_promote(bt, n_phys, promoted, evicted, hk, hv, kp, vp, T)
    assert err == 0 and moved == len(promoted)
    q = bf16_bits(rng, (G, D))
    # the pool after promotion, through the table
    out_a, lse_a, e1 = oracle_mod.unit_sparse_attention(q, kp.reshape(-1), vp.reshape(-1), T, bt, seq, cur)
    # the host store itself as the pool, identity table
    ident = np.arange(Pmax, dtype=np.int32)
    out_b, lse_b, e2 = oracle_mod.unit_sparse_attention(q, hk.reshape(-1), hv.reshape(-1), T, ident, seq, cur)
    assert e1 == 0 and e2 == 0
    assert np.array_equal(out_a, out_b) and np.array_equal(lse_a, lse_b)


def test_surplus_pages_and_blocks(oracle_mod):
    rng = np.random.default_rng(7)
    # more promoted than evicted: the last promoted page finds no block
    prev, cur = [2, 4, 6], [2, 5, 7, 9]
    hk, hv, bt, kp, vp, n_phys = resident_unit(rng, 12, prev)
    promoted, evicted = diff_lists(prev, cur)  # [5, 7, 9], [4, 6]
    err, moved, freed = oracle_mod.unit_promote(bt, n_phys, promoted, evicted, hk, hv, kp, vp, T)
    assert err == 0 and moved == 2 and len(freed) == 0
    assert (bt[promoted[:2]] >= 0).all() and bt[9] == -1
    # more evicted than promoted: surplus blocks come back in evicted order
    prev, cur = [1, 3, 8, 10], [1, 5]
    hk, hv, bt, kp, vp, n_phys = resident_unit(rng, 12, prev)
    blocks = bt.copy()
    promoted, evicted = diff_lists(prev, cur)  # [5], [3, 8, 10]
    err, moved, freed = oracle_mod.unit_promote(bt, n_phys, promoted, evicted, hk, hv, kp, vp, T)
    assert err == 0 and moved == 1
    assert freed.tolist() == [blocks[8], blocks[10]] and bt[5] == blocks[3]
    assert (bt[[3, 8, 10]] == -1).all()


def test_a_null_evicted_entry_is_reported_and_moves_nothing(oracle_mod):
    rng = np.random.default_rng(8)
    prev, cur = [1, 2], [1, 6]
    hk, hv, bt, kp, vp, n_phys = resident_unit(rng, 10, prev)
    bt[2] = -1  # the evicted page was already null
    err, moved, _ = oracle_mod.unit_promote(bt, n_phys, [6], [2], hk, hv, kp, vp, T)
    assert err & 1 and moved == 0 and bt[6] == -1


def test_table_update_applies_exactly_the_changed_entries(oracle_mod):
    # FlexiCache, "System design, head-level block table" (dirty tracking): the entries where two tables differ,
    # applied to the first, give the second; invalid updates are skipped and reported
    rng = np.random.default_rng(9)
    old = rng.integers(-1, 500, size=(2, 3, 4, 64)).astype(np.int32)
    new = old.copy()
    pick = rng.random(new.shape) < 0.05
    new[pick] = rng.integers(-1, 500, size=int(pick.sum()))
    idx = np.flatnonzero(old != new)
    t = old.copy()
    assert oracle_mod.table_update(t, 500, idx, new.ravel()[idx]) == 0
    assert np.array_equal(t, new)
    t2 = old.copy()
    err = oracle_mod.table_update(t2, 500, np.array([0, old.size, 5], dtype=np.int64), np.array([7, 1, 500], dtype=np.int32))
    assert err == 2 and t2.ravel()[0] == 7 and np.array_equal(t2.ravel()[1:], old.ravel()[1:])
