"""Pins of the oracle's mean-key scorer and dense page mass.

KVDrive, "Method details": each page's mean key is its representative in the
index, and pages are ranked by the query against it.  The pins: a page of
identical rows has that row as mean; the bf16 rounding equals torch's
nearest-even conversion of the fp32 mean; a unit-vector query reads one
channel; on single-token pages the MinMax bound (FlexiCache, "Core method,
2") and the mean-key score coincide, which ties the two scorers together;
the dense attention mass of the pages sums to 1 and is uniform for zero
keys.
"""
import numpy as np
import pytest
import torch


T, D = 16, 64




def bits(x):
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_identical_rows_average_to_themselves(oracle_mod):
    rng = np.random.default_rng(1)
    row = bits(rng.standard_normal(D))
    k = np.tile(row, (T, 1))
    mean, err = oracle_mod.unit_meankey(k.reshape(1, T, D), T, [0], T)
    assert err == 0 and np.array_equal(mean[0], row)


def test_rounding_is_torchs_nearest_even_of_the_fp32_mean(oracle_mod):
    rng = np.random.default_rng(2)
    for n in (1, 2, 3, 7, 16):
        k = bits(rng.standard_normal((T, D)) * 3)
        mean, _ = oracle_mod.unit_meankey(k.reshape(1, T, D), T, [0], n)
        vals = torch.tensor(k.view(np.int16)).view(torch.bfloat16).float()[:n]
        acc = torch.zeros(D, dtype=torch.float32)
        for r in range(n):  # fp32, token order
            acc = acc + vals[r]
        want = (acc / n).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(mean[0], want)
    # an exact tie between two bf16 neighbours rounds to the even one
    k = bits(np.stack([np.full(D, 1.0), np.full(D, 1.0078125)]))
    mean, _ = oracle_mod.unit_meankey(np.concatenate([k, np.zeros((T - 2, D), np.uint16)]).reshape(1, T, D), T, [0], 2)
    assert (mean[0] == bits(np.full(D, 1.0))).all()


def test_unit_query_reads_one_channel_and_single_token_pages_agree_with_minmax(oracle_mod):
    rng = np.random.default_rng(3)
    P = 12
    k = bits(rng.standard_normal((P, T, D)))
    seq = P * T
    mean, _ = oracle_mod.unit_meankey(k, T, np.arange(P), seq)
    q = np.zeros((1, D), dtype=np.float32)
    q[0, 5] = 1.0
    s = oracle_mod.unit_mean_scores(bits(q), mean, P)
    assert np.array_equal(s, torch.tensor(mean[:, 5].view(np.int16)).view(torch.bfloat16).double().numpy())
    # one token per page: min = max = mean = the key, and both scores are q . k
    k1 = k.copy()
    k1[:, 1:, :] = 0
    seq1 = (P - 1) * T + 1  # the last page holds one token
    qg = bits(rng.standard_normal((4, D)))
    m1, _ = oracle_mod.unit_meankey(k1, T, np.arange(P), seq1)
    mm, _ = oracle_mod.unit_minmax(k1, T, np.arange(P), seq1)
    s_mean = oracle_mod.unit_mean_scores(qg, m1, P)
    s_mm = oracle_mod.unit_scores(qg, mm, P)
    assert s_mean[-1] == pytest.approx(s_mm[-1], rel=1e-12)


def test_page_mass_sums_to_one_and_is_uniform_for_zero_keys(oracle_mod):
    rng = np.random.default_rng(4)
    P, seq = 9, 9 * T - 5
    k = bits(rng.standard_normal((P, T, D)))
    q = bits(rng.standard_normal((3, D)))
    mass = oracle_mod.unit_page_mass(q, k, T, np.arange(P), seq)
    assert mass.shape == (3, P) and np.allclose(mass.sum(axis=1), 1.0, atol=1e-12)
    zero = np.zeros_like(k)
    mz = oracle_mod.unit_page_mass(q, zero, T, np.arange(P), seq)
    want = np.array([min(T, seq - p * T) for p in range(P)], dtype=np.float64) / seq
    assert np.allclose(mz, want[None, :], atol=1e-15)
