"""Byte accounting against the figures the pages print (tests/golden/page_figures.txt)."""
import os

from paged_kv_cache_minmax_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.txt")


def load_figures():
    figs = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, value, unit, _src = [x.strip() for x in line.split("|", 3)]
        figs[name] = (float(value), unit)
    return figs


def test_kv_bytes_per_token_of_the_llama3_8b_shape():
    value, unit = load_figures()["kv_bytes_per_token_llama3_8b"]
    assert unit == "bytes"
    cfg = workloads.CONFIGS[2]  # 32 layers, 8 KV heads, head_dim 128, bf16
    assert workloads.kv_bytes_per_token(cfg.L, cfg.Hkv, cfg.D) == value


def test_stable_head_topk_volume_at_2048_token_budget():
    value, unit = load_figures()["stable_topk_bytes_llama31_8b_budget2048"]
    assert unit == "MiB"
    cfg = workloads.CONFIGS[2]
    stable_fraction = 0.75
    budget_tokens = cfg.K * cfg.T  # 128 pages of 16 tokens
    assert budget_tokens == 2048
    total = budget_tokens * workloads.kv_bytes_per_token(cfg.L, cfg.Hkv, cfg.D) * stable_fraction
    assert total / 2**20 == value
