"""Pins of the oracle's centroid level (KVDrive, "Method details": the pages' mean keys grouped under
higher-level centroids by similarity; "the trade-off between block size and centroid count").

Each pin checks the oracle against something other than itself: exact arithmetic on integer-valued keys,
closed forms (identical pages, one page a centroid, every centroid expanded equals the flat mean-key
search), properties of each Lloyd step recomputed independently in float64 (each page joins a nearest
centroid; each centroid is the mean of its members), and a planted two-group layout that similarity
grouping must separate where spatial blocks mix it.
"""
import numpy as np
import torch


def bits(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def vals(b):
    return torch.from_numpy(np.asarray(b, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).double().numpy()


def check_partition(P, off, members, assign):
    n_c = len(off) - 1
    assert off[0] == 0 and off[-1] == P and np.all(np.diff(off) >= 0)
    assert sorted(members.tolist()) == list(range(P))
    for j in range(n_c):
        grp = members[off[j]:off[j + 1]]
        assert np.all(np.diff(grp) > 0), "a group's pages are ascending"
        assert np.all(assign[grp] == j)


def test_identical_pages_make_identical_centroids(oracle_mod):
    row = bits(np.linspace(-3, 3, 64))
    mean = np.tile(row, (29, 1))
    for R, n_iter in ((1, 0), (4, 0), (4, 3), (7, 2)):
        cent, assign, off, members = oracle_mod.centroid_build(mean, R, n_iter)
        assert cent.shape == ((29 + R - 1) // R, 64)
        assert np.array_equal(cent, np.tile(row, (len(cent), 1)))
        check_partition(29, off, members, assign)
        if n_iter:
            assert np.all(assign == 0), "equal distances: the lowest centroid wins every tie"


def test_spatial_blocks_average_their_pages_exactly(oracle_mod):
    # integer keys: sums are exact in fp32, and a block of 4 divides exactly; the last block has 3 pages
    rs = np.random.default_rng(1)
    P, D, R = 23, 32, 4
    ints = rs.integers(-8, 9, size=(P, D)).astype(np.float64)
    cent, assign, off, members = oracle_mod.centroid_build(bits(ints), R, 0)
    assert assign.tolist() == [p // R for p in range(P)]
    check_partition(P, off, members, assign)
    for j in range(len(cent)):
        block = ints[j * R:(j + 1) * R]
        want = block.mean(axis=0)
        got = vals(cent[j])
        # exact where the mean is a bf16 value (every full block: quarters of small integers)
        if len(block) == R:
            assert np.array_equal(got, want)
        else:
            assert np.allclose(got, want, rtol=2 ** -8, atol=0)


def test_each_lloyd_step_assigns_nearest_and_averages_members(oracle_mod):
    rs = np.random.default_rng(2)
    P, D, R = 61, 64, 5
    mean = bits(rs.normal(size=(P, D)) * rs.uniform(0.5, 4, size=D))
    for k in range(3):
        c_k, _, _, _ = oracle_mod.centroid_build(mean, R, k)
        c_next, a_next, off, members = oracle_mod.centroid_build(mean, R, k + 1)
        check_partition(P, off, members, a_next)
        x, c = vals(mean), vals(c_k)
        dist = ((x[:, None, :] - c[None, :, :]) ** 2).sum(axis=2)  # float64, independent of the oracle's fp32
        best = dist.min(axis=1)
        for p in range(P):
            # the page's centroid is a nearest one (fp32 against float64: a relative margin)
            assert dist[p, a_next[p]] <= best[p] * (1 + 1e-5) + 1e-30, p
            # and no lower-indexed centroid is strictly nearer (ties go to the lower centroid)
            lower = dist[p, :a_next[p]]
            assert np.all(lower >= best[p] * (1 - 1e-5)), p
        # the new centroids: each the mean of its members (bf16 rounding), an empty one keeps its value
        cn = vals(c_next)
        for j in range(len(c_next)):
            grp = members[off[j]:off[j + 1]]
            if len(grp) == 0:
                assert np.array_equal(c_next[j], c_k[j])
            else:
                assert np.allclose(cn[j], x[grp].mean(axis=0), rtol=2 ** -7, atol=1e-6)


def test_similarity_grouping_separates_what_spatial_blocks_mix(oracle_mod):
    # two groups of pages near +u and -u; every spatial block of 4 holds three pages of one group and one of
    # the other (the majority alternating block by block), so each block's centroid leans to its majority:
    # after Lloyd steps each centroid holds pages of one group only.  u is a random direction, then the
    # first channel alone, then the last channel alone (so every channel takes part in the distance)
    rs = np.random.default_rng(3)
    P, D = 40, 64
    major = np.where((np.arange(P) // 4) % 2 == 0, 1.0, -1.0)
    sign = np.where(np.arange(P) % 4 == 3, -major, major)
    for u in (rs.normal(size=D), np.eye(D)[0], np.eye(D)[D - 1]):
        u = u / np.linalg.norm(u)
        noise = 0.05 * rs.normal(size=(P, D)) * (1 - np.abs(u) if np.count_nonzero(u) == 1 else 1)
        mean = bits(sign[:, None] * 3 * u[None, :] + noise)
        cent0, a0, _, _ = oracle_mod.centroid_build(mean, 4, 0)
        assert all(len(set(sign[a0 == j])) == 2 for j in range(len(cent0))), "spatial blocks mix both groups"
        # a centroid of a mixed block sits near 0; assigning pulls each page to the nearest centroid
        cent, assign, off, members = oracle_mod.centroid_build(mean, 4, 2)
        for j in range(len(cent)):
            grp = members[off[j]:off[j + 1]]
            assert len(set(sign[grp])) <= 1, "a centroid holds pages of one group"


def test_expanding_every_centroid_is_the_flat_mean_key_search(oracle_mod):
    rs = np.random.default_rng(4)
    P, D, G, K = 50, 64, 4, 9
    mean = bits(rs.normal(size=(P, D)))
    q = bits(rs.normal(size=(G, D)))
    cent, _, off, members = oracle_mod.centroid_build(mean, 6, 2)
    for group_reduce in (0, 1):
        r = oracle_mod.centroid_select(q, mean, cent, off, members, M=len(cent), K=K, group_reduce=group_reduce)
        flat = oracle_mod.topk(oracle_mod.unit_mean_scores(q, mean, P, group_reduce), K)
        assert r["cand"].tolist() == list(range(P))
        assert r["sel"].tolist() == flat.tolist()


def test_one_page_a_centroid_scores_centroids_as_pages(oracle_mod):
    rs = np.random.default_rng(5)
    P, D, G, K = 30, 64, 2, 6
    mean = bits(rs.normal(size=(P, D)))
    q = bits(rs.normal(size=(G, D)))
    cent, assign, off, members = oracle_mod.centroid_build(mean, 1, 0)
    assert np.array_equal(cent, mean) and assign.tolist() == list(range(P))
    r = oracle_mod.centroid_select(q, mean, cent, off, members, M=K, K=K)
    assert np.array_equal(r["cs"], oracle_mod.unit_mean_scores(q, mean, P))
    assert r["sel"].tolist() == r["chosen"].tolist() == oracle_mod.topk(r["cs"], K).tolist()


def test_selection_keeps_the_best_pages_of_the_chosen_centroids(oracle_mod):
    rs = np.random.default_rng(6)
    P, D, G = 80, 64, 4
    mean = bits(rs.normal(size=(P, D)))
    q = bits(rs.normal(size=(G, D)))
    cent, _, off, members = oracle_mod.centroid_build(mean, 8, 1)
    r = oracle_mod.centroid_select(q, mean, cent, off, members, M=3, K=7)
    # the chosen centroids are the 3 best by q . c; the candidates are exactly their pages
    cs = vals(cent) @ vals(q).T
    assert r["chosen"].tolist() == sorted(np.argsort(-cs.sum(axis=1), kind="stable")[:3].tolist())
    cand = sorted(p for j in r["chosen"] for p in members[off[j]:off[j + 1]])
    assert r["cand"].tolist() == cand
    # the selection: the 7 best candidates by q . mean (sum over heads), ascending
    ps = (vals(mean)[cand] @ vals(q).T).sum(axis=1)
    best = sorted(np.array(cand)[np.argsort(-ps, kind="stable")[:7]].tolist())
    assert r["sel"].tolist() == best
    # K beyond the candidates: all of them
    r2 = oracle_mod.centroid_select(q, mean, cent, off, members, M=2, K=10 ** 6)
    assert r2["sel"].tolist() == r2["cand"].tolist()
