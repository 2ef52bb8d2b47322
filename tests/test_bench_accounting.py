"""bench.py's byte accounting, the numerator of every GB/s and roofline figure it reports.

Checked against the sizes the workloads fix: MinMax rows of every page of
every rescored unit, K and V of every selected page, and small terms well
under 1% at the full-size shapes.
"""
import bench
from paged_kv_cache_minmax_gb300 import workloads


def test_llama8b_32k_layer_step_moves_64_mib_of_metadata_and_64_mib_of_selected_kv():
    cfg = workloads.CONFIGS[2]
    b = bench.algorithmic_bytes(cfg)
    units = cfg.B * cfg.Hkv  # 64
    assert b["meta"] == units * cfg.P * 2 * cfg.D * 2 == 64 * 2**20
    assert b["kv"] == units * cfg.K * cfg.T * cfg.D * 2 * 2 == 64 * 2**20
    assert 0 < b["small"] < 0.01 * b["total"]
    assert b["total"] == b["meta"] + b["kv"] + b["small"]
    # one decode_layer launch: the metadata and pages, plus its own small terms
    assert b["meta"] + b["kv"] < b["decode_launch"] < 1.01 * (b["meta"] + b["kv"])


def test_the_rerank_schedule_counts_only_rescored_units_metadata():
    cfg = workloads.CONFIGS[4]
    all_units = cfg.B * cfg.Hkv
    full = bench.algorithmic_bytes(cfg)
    quarter = bench.algorithmic_bytes(cfg, rescored_units=all_units / 4)
    assert quarter["kv"] == full["kv"]  # every unit attends over its selection every step
    assert quarter["meta"] == full["meta"] / 4
    assert quarter["total"] < full["total"]


def test_k_at_least_p_selects_every_page():
    cfg = workloads.scaled(workloads.CONFIGS[1], K=10**6)
    b = bench.algorithmic_bytes(cfg)
    assert b["kv"] == cfg.B * cfg.Hkv * cfg.P * cfg.T * cfg.D * 2 * 2


def test_measured_traffic_is_reported_only_for_the_captured_workload_batch_and_sources(tmp_path, monkeypatch):
    import json
    import os

    from paged_kv_cache_minmax_gb300 import build as kbuild

    # the committed captures: one launch of each workload, within a few percent of its algorithmic bytes
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        committed = json.load(f)
    for c in (2, 3, 5):
        cfg = workloads.CONFIGS[c]
        rec = committed["decode_layer"][cfg.name]
        launch = bench.algorithmic_bytes(cfg)["decode_launch"]
        assert rec["batch"] == cfg.B and launch <= rec["bytes"] < 1.05 * launch, c
    # the gate: the workload, its batch and the sources the capture was taken with
    name = workloads.CONFIGS[2].name
    B = workloads.CONFIGS[2].B
    (tmp_path / "profiles").mkdir()
    with open(tmp_path / "profiles" / "traffic.json", "w") as f:
        json.dump({"decode_layer": {name: {"batch": B, "bytes": 123, "sources": kbuild.source_digest()}},
                   "page_score_topk": {name: {"batch": B, "bytes": 456, "sources": "0000000000000000"}}}, f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("decode_layer", name, B) == 123
    assert bench.load_traffic("decode_layer", name, 4) is None  # another batch: another launch
    assert bench.load_traffic("decode_layer", workloads.CONFIGS[4].name, workloads.CONFIGS[4].B) is None
    assert bench.load_traffic("sparse_attn_kernel", name, B) is None
    assert bench.load_traffic("page_score_topk", name, B) is None  # taken with other sources


def test_the_mix_episode_counts_the_units_each_step_rescores():
    """The stable/unstable episode: every unit on a rerank step, else the batch times a layer's unstable heads
    (on average over the layers); a layer-step's bytes follow."""
    cfg = workloads.scaled(workloads.CONFIGS[4], B=2, L=4, S=256, K=8, steps=32, n_planted=4)
    wl = workloads.generate(cfg, device="cpu")
    ep = bench.MixEpisode(wl, None)
    n_unstable = int(wl.unstable.sum())
    assert n_unstable == round(0.25 * cfg.L * cfg.Hkv)
    assert ep.rerank(0) and ep.rerank(16) and not ep.rerank(1)
    assert ep.mask(0) is None and ep.mask(5) is ep.unstable
    assert ep.rescored_units(0, cfg.B) is None
    assert ep.rescored_units(3, cfg.B) == cfg.B * n_unstable / cfg.L
    between = bench.algorithmic_bytes(cfg, rescored_units=ep.rescored_units(3, cfg.B))
    full = bench.algorithmic_bytes(cfg)
    assert between["meta"] == full["meta"] * n_unstable / (cfg.L * cfg.Hkv)
    # the episode's inputs: one appended token per step at the sequence's end
    assert ep.seq.shape == (cfg.steps, cfg.B) and int(ep.seq[0, 0]) == cfg.S + 1
    assert ep.tb[5].tolist() == (ep.seq[5] - 1).tolist()
