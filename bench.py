"""Benchmark: MinMax page selection + sparse paged decode attention on GB300.

One step = one decode step of the Llama-3.1-8B-shaped 32K-context workload
(32 layers, B=8, 32 query / 8 KV heads, head_dim 128, 16-token pages,
budget 128 pages): per layer, append the new token and refresh its page's
MinMax, score every page, select the top-K and attend over the selected
pages -- decode_layer, one launch -- and list promoted pages
(topk_promotion_diff, on a side stream).  --path fused runs
kv_minmax_update and page_score_topk_attn (one launch that scores, selects
and attends) instead; --path unfused runs kv_minmax_update, page_score_topk
and sparse_paged_decode_attn.  A
layer-step is one layer of that step for the whole batch.

Inputs are seeded synthetic tensors resident in HBM (32 GiB of K/V, 2 GiB of
metadata); one step touches 4 GiB of distinct data, far more than the 129 MB
L2, so no flush is needed between steps.  The step is captured once in a
CUDA graph and replayed; CUDA events on the launching stream time the timed
region and every launch of the decode (or scoring and attention) kernels.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_minmax_gb300 import workloads  # noqa: E402

METRIC = "sparse decode attn+scoring: KV GB/s & % of HBM peak; layer-steps/s at 32K ctx"
CFG = workloads.CONFIGS[2]
FALLBACK_HBM_GBS = 6800.0


# --------------------------------------------------------------------------- #
# byte accounting                                                              #
# --------------------------------------------------------------------------- #
def algorithmic_bytes(cfg, rescored_units=None):
    """Bytes one layer-step must move at minimum (all units of one layer).

    meta   : MinMax rows of every page of every rescored unit (P * 2 * D * 2 B)
    kv     : K and V rows of every selected page (K * T * D * 2 B each)
    small  : q, selected table entries, selection lists (write + read), the
             promotion diff, outputs, the appended token and its page's
             re-read and metadata write.
    """
    units = cfg.B * cfg.Hkv
    resc = units if rescored_units is None else rescored_units
    P, K = cfg.P, min(cfg.K, cfg.P)
    meta = resc * P * 2 * cfg.D * 2
    kv = units * K * cfg.T * cfg.D * 2 * 2
    page = cfg.T * cfg.D * 2
    small = (cfg.B * cfg.Hq * cfg.D * 2 * 2          # q read by scoring and by attention
             + units * K * 4                          # table entries of selected pages
             + units * K * 4 * 3                      # selection written, read by diff and attention
             + resc * K * 4 * 3                       # prev read, promoted written, prev committed
             + cfg.B * cfg.Hq * (cfg.D + 1) * 4       # out + lse
             + units * (2 * cfg.D * 2 + page + 2 * cfg.D * 2))  # new K/V row, page re-read, meta write
    return {"meta": meta, "kv": kv, "small": small, "total": meta + kv + small,
            "score_launch": meta + cfg.B * cfg.Hq * cfg.D * 2 + units * K * 4,
            "attn_launch": kv + cfg.B * cfg.Hq * cfg.D * 2 + units * K * 8 + cfg.B * cfg.Hq * (cfg.D + 1) * 4,
            # one launch: metadata, selected K/V, q, table entries, selection written and read, out + lse
            "fused_launch": meta + kv + cfg.B * cfg.Hq * cfg.D * 2 + units * K * 4 * 3
                            + cfg.B * cfg.Hq * (cfg.D + 1) * 4,
            # decode_layer: the above, plus the append (new K/V row read, the page's earlier rows re-read,
            # its metadata row written)
            "decode_launch": meta + kv + cfg.B * cfg.Hq * cfg.D * 2 + units * K * 4 * 3
                             + cfg.B * cfg.Hq * (cfg.D + 1) * 4 + units * (2 * cfg.D * 2 + page + 2 * cfg.D * 2)}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# --------------------------------------------------------------------------- #
# clocks during the timed region                                               #
# --------------------------------------------------------------------------- #
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0, out_path=None):
        self.out_path = out_path
        self.proc = None
        self.device_index = device_index

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
            if self.out_path:
                with open(self.out_path, "w") as f:
                    f.write(self.FIELDS + "\n" + "\n".join(self.lines) + "\n")

    def summary(self):
        if not getattr(self, "lines", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- #
# CPU oracle timing (cpu_baseline and the reference arm)                      #
# --------------------------------------------------------------------------- #
def oracle_layer_sample(cfg, n_units, seed=2024, device=None):
    """Host state for ``n_units`` units of one layer of ``cfg`` (compact pools)."""
    import oracle

    sub = workloads.scaled(cfg, B=max(1, -(-n_units // cfg.Hkv)), L=1, layers_alloc=None)
    dev = device or ("cuda" if torch.cuda.is_available() else "cpu")
    wl = workloads.generate(sub, device=dev, seed=seed)
    nk, nv = workloads.step_tokens(wl, 0)
    states = []
    for u in range(n_units):
        b, h = divmod(u, sub.Hkv)
        row = wl.block_table[b, 0, h].cpu().numpy().astype(np.int32)
        idx = torch.as_tensor(row[: sub.Pmax], dtype=torch.long, device=wl.k_pool.device)
        kp = workloads.bf16_bits(wl.k_pool.index_select(0, idx))
        vp = workloads.bf16_bits(wl.v_pool.index_select(0, idx))
        local = np.arange(sub.Pmax, dtype=np.int32)
        meta, _ = oracle.unit_minmax(kp, sub.T, local, int(wl.seq_len[b]))
        stt = oracle.UnitState(kp, vp, sub.T, local, meta, sub.K)
        qg = workloads.bf16_bits(wl.q[0, b, h * sub.G:(h + 1) * sub.G])
        states.append((stt, int(wl.seq_len[b]), workloads.bf16_bits(nk[0, b, h]), workloads.bf16_bits(nv[0, b, h]),
                       qg))
    del wl
    return states


def run_oracle_units(states, threads):
    """One decode step (rescored) of every unit in ``states``; returns seconds."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    def one(s):
        stt, seq, nk, nv, qg = s
        oracle.unit_step(stt, seq, nk, nv, qg, rescore=True)

    t0 = time.perf_counter()
    if threads <= 1:
        for s in states:
            one(s)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, states))
    return time.perf_counter() - t0


def cpu_baseline(cfg, target_seconds=12.0):
    """The oracle on the host cores over whole layer-steps: every (batch, KV head) unit of one layer, each
    unit's own pages (no unit's data stays cached for the next layer-step), repeated for about
    ``target_seconds`` of wall time."""
    import oracle

    oracle.build()
    threads = os.cpu_count() or 1
    units_per_layer = cfg.B * cfg.Hkv
    states = oracle_layer_sample(cfg, units_per_layer)
    first = run_oracle_units(states, threads)  # one layer-step (also warms the code)
    reps = max(1, int(target_seconds / max(first, 1e-6)))
    wall = sum(run_oracle_units(states, threads) for _ in range(reps))
    ls_per_s = reps / wall
    one = run_oracle_units(states, 1)  # the same layer-step on one thread
    b = algorithmic_bytes(cfg)
    return {"value": ls_per_s, "unit": "layer-steps/s", "cores": threads, "kind": "oracle",
            "gbs": b["total"] * ls_per_s / 1e9,
            "one_thread": {"value": 1.0 / one, "unit": "layer-steps/s", "gbs": b["total"] / one / 1e9,
                           "sample": "one layer-step on one thread"},
            "sample": f"{reps} layer-steps of {cfg.name}, each all {units_per_layer} (batch, KV head) units of one "
                      f"layer (per unit: append+MinMax, score all {cfg.P} pages, top-{cfg.K}, diff, attention), "
                      f"on {threads} threads; {wall:.1f} s wall"}


def reference_arm(args):
    """The oracle, as it stands, on the host cores: the slow reference program."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    cfg = workloads.CONFIGS[args.config]
    threads = os.cpu_count() or 1
    units = cfg.B * cfg.Hkv
    states = oracle_layer_sample(cfg, units)
    for _ in range(args.warmup):
        run_oracle_units(states, threads)
    times = [run_oracle_units(states, threads) for _ in range(args.steps)]
    total = sum(times)
    value = args.steps / total  # layer-steps per second
    b = algorithmic_bytes(cfg)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; stands in for Llama-3.1-8B long-context decode)",
            "config": {"workload": cfg.name, "layer_step": f"one layer of one decode step, {units} units",
                       "global_batch": cfg.B, "seq_len": cfg.S, "top_k_pages": cfg.K, "page_tokens": cfg.T},
            "kv_gbs": b["total"] * value / 1e9,
            "cpu_baseline": {"kind": "oracle", "cores": threads, "value": value, "unit": "layer-steps/s",
                             "sample": f"each step = all {units} units of one layer (C oracle, double "
                                       f"precision) on {threads} threads"},
            "e2e": {"value": value, "unit": "layer-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# GPU arm                                                                      #
# --------------------------------------------------------------------------- #
def replica_seed(cfg, rank):
    """Replicas: every rank decodes its own batch of the workload, seeded apart (no data-path collective)."""
    return cfg.seed + 7919 * rank


def max_over_ranks(value, dist, device):
    """The slowest rank's time: a replica job ends when its last rank does (the value is unchanged alone)."""
    if dist is None:
        return value
    t = torch.tensor([float(value)], device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t)


def make_timing_events(n):
    try:
        return [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)], True
    except TypeError:
        return [torch.cuda.Event(enable_timing=True) for _ in range(n)], False


def decode_layer_call(st, l, q, nk, nv, early_reads, mask=None, tok_begin=None, seq_len=None):
    """decode_layer for layer ``l`` as the bench launches it: one new token per sequence written at
    ``tok_begin`` (the sequence's last position; ``seq_len`` counts it), every page of the rescored units
    scored, K selected, attention over them."""
    tb = st.tok_begin if tok_begin is None else tok_begin
    sl = st.seq_len if seq_len is None else seq_len
    kvmm = _kvmm()
    kvmm.decode_layer(st.shape, l, q, nk, nv, 1, tb, sl, st.k_pool, st.v_pool, st.block_table, st.meta, sl, mask,
                      st.K, st.sel_idx, st.sel_cnt, st.out[l], lse=st.lse[l], err=st.err, workspace=st.workspace,
                      early_reads=early_reads)


def decode_step(st, path, L, q, nk, nv, early_reads, side, forks, mask=None, ev=None, tok_begin=None,
                seq_len=None, total_promoted=None):
    """One decode step exactly as the bench times it.  Per layer l: decode_layer (path "decode_layer"), or
    kv_minmax_update and then page_score_topk_attn ("fused") or page_score_topk and sparse_paged_decode_attn
    ("unfused"); and topk_promotion_diff on the stream ``side``, forked after the layer's selection and joined
    at the end of the step.  q [L][B][Hq][D], nk / nv [L][B][Hkv][1][D]; ``ev``: 4 events a layer bracketing
    the selection (or decode) launch and the attention launch."""
    kvmm = _kvmm()
    main = torch.cuda.current_stream()
    tb = st.tok_begin if tok_begin is None else tok_begin
    sl = st.seq_len if seq_len is None else seq_len
    tp = st.total_promoted if total_promoted is None else total_promoted
    for l in range(L):
        if path != "decode_layer":
            kvmm.kv_minmax_update(st.shape, l, nk[l], nv[l], 1, tb, sl, st.k_pool, st.v_pool, st.block_table,
                                  st.meta, st.err)
        if ev is not None:
            ev[4 * l].record()
        if path == "decode_layer":  # append, score, select and attend in one launch
            decode_layer_call(st, l, q[l], nk[l], nv[l], early_reads, mask, tb, sl)
        elif path == "fused":  # scoring, then attention that selects its own pages
            kvmm.page_score_topk_attn(st.shape, l, q[l], st.meta, st.k_pool, st.v_pool, st.block_table, sl, mask,
                                      st.K, st.sel_idx, st.sel_cnt, st.out[l], st.workspace, lse=st.lse[l],
                                      err=st.err)
        else:
            kvmm.page_score_topk(st.shape, l, q[l], st.meta, sl, mask, st.K, st.sel_idx, st.sel_cnt, st.workspace,
                                 st.err)
        if ev is not None:
            ev[4 * l + 1].record()
        forks[l].record(main)
        side.wait_event(forks[l])
        with torch.cuda.stream(side):
            kvmm.topk_promotion_diff(st.shape, l, mask, st.prev_idx, st.prev_cnt, st.sel_idx, st.sel_cnt,
                                     st.promoted, st.promoted_cnt, st.evicted, st.evicted_cnt, tp, commit=True,
                                     err=st.err)
        if path == "unfused":
            if ev is not None:
                ev[4 * l + 2].record()
            # early reads: the scoring call just before writes selections and scores only (it reads early
            # nothing itself: the update before it writes the metadata rows it scores)
            kvmm.sparse_paged_decode_attn(st.shape, l, q[l], st.k_pool, st.v_pool, st.block_table, sl, st.sel_idx,
                                          st.sel_cnt, st.out[l], st.workspace, lse=st.lse[l], err=st.err,
                                          num_splits=st.num_splits, early_reads=early_reads)
            if ev is not None:
                ev[4 * l + 3].record()
    main.wait_stream(side)


def _kvmm():
    from paged_kv_cache_minmax_gb300 import kvmm

    return kvmm


class MixEpisode:
    """The stable/unstable workload's decode episode (64 steps): step t appends one token per sequence at
    position S + t, with queries drifting as q_t = 0.9 q_{t-1} + 0.44 eps, and rescores every unit when
    t % rerank_period == 0, else only the unstable heads' units (the others keep their selection).  Every
    step's inputs sit in buffers of their own, so each step is one CUDA graph; after the last step the
    episode starts over at position S (those tokens are written again with the same values)."""

    def __init__(self, wl, st):
        cfg = wl.cfg
        self.E = cfg.steps
        self.period = cfg.rerank_period
        self.q = workloads.drift_queries(wl, self.E)  # [E, L, B, Hq, D]
        toks = [workloads.step_tokens(wl, t) for t in range(self.E)]
        self.nk = torch.stack([k for k, _ in toks]).contiguous()  # [E, L, B, Hkv, 1, D]
        self.nv = torch.stack([v for _, v in toks]).contiguous()
        base = wl.seq_len.clone()
        self.seq = torch.stack([base + t + 1 for t in range(self.E)]).contiguous()  # [E, B], after the append
        self.tb = (self.seq - 1).contiguous()
        self.unstable = wl.unstable.contiguous()
        self.prom = torch.zeros(self.E, dtype=torch.int32, device=wl.q.device)  # promoted pages per step

    def rerank(self, t):
        return t % self.period == 0

    def mask(self, t):
        return None if self.rerank(t) else self.unstable

    def rescored_units(self, t, B):
        """Units of one layer-step rescored at step t (None: all): on average over the layers, the batch times
        the unstable heads of a layer."""
        return None if self.rerank(t) else float(self.unstable.sum()) * B / self.unstable.shape[0]


def promotion_stats(ep, st, graphs, stream, K, B):
    """One pass over the episode from an empty selection, step by step: the pages topk_promotion_diff lists
    per step, split by rerank steps (every unit rescored) and the steps between (unstable heads only), and
    by stable and unstable heads, as a fraction of the K pages of the units that were rescored."""
    st.prev_cnt.zero_()
    st.sel_cnt.zero_()
    torch.cuda.synchronize()  # zeroed on the default stream; the steps replay on `stream`
    unst = ep.unstable.bool()[None, :, :].expand(B, -1, -1)  # [B, L, Hkv]
    per_step = []
    acc = {"rerank_stable": [0, 0], "rerank_unstable": [0, 0], "between_unstable": [0, 0]}
    for t in range(ep.E):
        with torch.cuda.stream(stream):
            graphs[t].replay()
        stream.synchronize()
        pc = st.promoted_cnt.clone()
        per_step.append(int(pc.sum()))
        if t == 0:
            continue  # the first selection promotes every page: not a rerank of a running decode
        if ep.rerank(t):
            for key, sel in (("rerank_stable", ~unst), ("rerank_unstable", unst)):
                acc[key][0] += int(pc[sel].sum())
                acc[key][1] += int(sel.sum()) * K
        else:
            acc["between_unstable"][0] += int(pc[unst].sum())
            acc["between_unstable"][1] += int(unst.sum()) * K
    frac = {k: (v[0] / v[1] if v[1] else None) for k, v in acc.items()}
    return {"promoted_per_step": per_step, "promoted_fraction_of_k": frac,
            "how": "one episode from an empty selection, step by step; step 0 (the first selection) is left out "
                   "of the fractions; a fraction is promoted pages / (rescored units x K)"}


def time_graphs(graph_list, stream, reps):
    """Mean ms of one replay of each graph: all replayed back to back ``reps`` times between two CUDA
    events on ``stream`` (after three untimed rounds)."""
    out = []
    for g in graph_list:
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        stream.synchronize()
        out.append(e0.elapsed_time(e1) / reps)
    return out


def separate_calls_leg(st, cfg, L, q_dev, stream, reps, peak):
    """page_score_topk alone, sparse_paged_decode_attn alone (over the selection the first leaves) and the
    two back to back, each as L launches of one CUDA graph replayed back to back (every unit rescored, the
    automatic split count).  Per launch: CUDA-event time and the algorithmic bytes of that call.  Both calls
    read early (KVMM_EARLY_READS): in every sequence timed here the launch before writes nothing they read
    early (scoring writes selections and scores; attention writes outputs; neither writes lengths, masks,
    tables or metadata)."""
    kvmm = _kvmm()

    def score(l):
        kvmm.page_score_topk(st.shape, l, q_dev[l], st.meta, st.seq_len, None, st.K, st.sel_idx, st.sel_cnt,
                             st.workspace, st.err, early_reads=True)

    def attn(l):
        kvmm.sparse_paged_decode_attn(st.shape, l, q_dev[l], st.k_pool, st.v_pool, st.block_table, st.seq_len,
                                      st.sel_idx, st.sel_cnt, st.out[l], st.workspace, lse=st.lse[l], err=st.err,
                                      num_splits=st.num_splits, early_reads=True)

    with torch.cuda.stream(stream):
        for l in range(L):
            score(l)
            attn(l)
    stream.synchronize()
    graphs = []
    for body in ((score,), (attn,), (score, attn)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(L):
                for fn in body:
                    fn(l)
        graphs.append(g)
    ms_s, ms_a, ms_p = (m / L for m in time_graphs(graphs, stream, reps))
    b = algorithmic_bytes(cfg)

    def rec(ms, nbytes, kernel=None):
        gbs = nbytes / (ms / 1e3) / 1e9
        out = {"us_per_launch": ms * 1e3, "bytes_per_launch": nbytes, "gbs": gbs, "frac": gbs / peak}
        if kernel is not None:  # DRAM bytes of one launch from the committed ncu capture, if there is one
            out["traffic"] = load_traffic(kernel, cfg.name, cfg.B)
        return out

    both = b["score_launch"] + b["attn_launch"]
    return {"page_score_topk": rec(ms_s, b["score_launch"], "page_score_topk"),
            "sparse_paged_decode_attn": rec(ms_a, b["attn_launch"], "sparse_paged_decode_attn"),
            "sum_of_alone": rec(ms_s + ms_a, both),
            "back_to_back": rec(ms_p, both),
            "flags": "KVMM_EARLY_READS",
            "how": f"{L} launches of each call (or {L} pairs) in one CUDA graph, replayed {reps} times between "
                   "CUDA events on the launching stream; per launch = region / launches; bytes per launch: "
                   "the call's metadata or selected K/V plus its small terms"}


def gpu_arm(args):
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm
    from paged_kv_cache_minmax_gb300.runtime import DecodeState

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    kbuild.build_library()
    kvmm.load()

    cfg = workloads.CONFIGS[args.config]
    if args.batch or args.layers:
        cfg = workloads.scaled(cfg, B=args.batch or cfg.B, L=args.layers or cfg.L)
    L = cfg.L_alloc  # a step rotates over the allocated layers
    # replicas: every rank decodes its own batch (seeded per rank); no collective on the data path
    wl = workloads.generate(cfg, device="cuda", seed=replica_seed(cfg, rank))
    shape = kvmm.make_shape(cfg.B, L, cfg.Hq, cfg.Hkv, cfg.D, cfg.T, cfg.Pmax, cfg.K, wl.n_phys)
    splits = kvmm.auto_splits(shape)
    st = DecodeState.for_workload(wl)  # automatic split count (0): the clustered attention kernel
    one_launch = True  # decode_layer runs its one-launch kernel (else its two-kernel fallback)
    clustered = kvmm.decode_layer_cluster(shape) > 0  # the shape fits the clustered decode kernel
    if args.path == "decode_layer":
        c_ctas = kvmm.decode_layer_cluster(shape)
        one_launch = c_ctas > 0
        launch_shape = ({"units_per_cluster": kvmm.decode_layer_units(shape), "cluster_ctas": c_ctas}
                        if one_launch else
                        {"splits": splits, "decode_layer": "falls back to kv_minmax_update + page_score_topk_attn "
                                                           "(per-CTA buffers exceed shared memory)"})
    else:
        launch_shape = {"splits": splits}
    path = args.path
    # the layers' decode_layer calls follow one another on the stream, and none writes what the next reads
    # of the cache state (its own layer's rows only; lengths and masks change between steps): each launch
    # may stream its metadata while the previous one drains (KVMM_DECODE_EARLY_READS).  With one allocated
    # layer consecutive calls are for the same layer, and the earlier one writes the metadata row the later
    # one would read early: the flag stays off there.
    early_reads = not args.no_early_reads and L >= 2
    st.build_metadata()
    stream = torch.cuda.Stream()
    side = torch.cuda.Stream()  # the promotion diff is not needed by attention: a side stream
    forks = [torch.cuda.Event() for _ in range(L)]
    ev_s, external = make_timing_events(4 * L)

    episode = cfg.steps > 0
    if episode:
        # the stable/unstable workload: a drifting decode episode, one graph per step
        ep = MixEpisode(wl, st)
        E = ep.E

        def step_inputs(t):
            return dict(q=ep.q[t], nk=ep.nk[t], nv=ep.nv[t], mask=ep.mask(t), tok_begin=ep.tb[t],
                        seq_len=ep.seq[t], total_promoted=ep.prom[t:t + 1])
    else:
        # one token per sequence at position seq_len - 1, written again every step with the same values
        E = 1
        nk0, nv0 = workloads.step_tokens(wl, 0)
        st.tok_begin.copy_(wl.seq_len - 1)
        q_dev, nk_dev, nv_dev = wl.q.clone(), nk0.clone(), nv0.clone()

        def step_inputs(t):
            return dict(q=q_dev, nk=nk_dev, nv=nv_dev)

    def run_step(t, ev=None):
        a = step_inputs(t)
        decode_step(st, path, L, a["q"], a["nk"], a["nv"], early_reads, side, forks, mask=a.get("mask"), ev=ev,
                    tok_begin=a.get("tok_begin"), seq_len=a.get("seq_len"), total_promoted=a.get("total_promoted"))

    torch.cuda.empty_cache()
    torch.cuda.synchronize()  # the set-up ran on the default stream; everything below runs on `stream`
    with torch.cuda.stream(stream):
        for t in range(min(3, E) if episode else 3):
            run_step(t)
    stream.synchronize()
    if args.no_graph:  # eager launches (profiling): same kernels, host-issued every step
        external = False

        class _Eager:
            def __init__(self, t):
                self.t = t

            def replay(self):
                run_step(self.t)

        graphs = [_Eager(t) for t in range(E)]
        graph_instr = None
    else:
        graphs = []
        for t in range(E):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                run_step(t)
            graphs.append(g)
        external = external and not episode  # the episode's roofline uses the graph below
        graph_instr = torch.cuda.CUDAGraph() if external else None
        if external:
            with torch.cuda.graph(graph_instr, stream=stream):
                run_step(0, ev_s)
    promotions = None
    if episode:  # first, the episode once from an empty selection, counting promotions
        promotions = promotion_stats(ep, st, graphs, stream, cfg.K, cfg.B)
    st.err.zero_()
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % E].replay()
    stream.synchronize()

    # ---- timed region (device-resident inputs) --------------------------------
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local_rank, args.clocks_log)
    timed_steps = [(args.warmup + i) % E for i in range(args.steps)]
    with clocks:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            t0.record()
            for i, t in enumerate(timed_steps):
                if external and i == args.steps - 1:
                    graph_instr.replay()  # the last step also stamps every kernel launch
                else:
                    graphs[t].replay()
            t1.record()
        stream.synchronize()
    torch.cuda.synchronize()
    ms_total = max_over_ranks(t0.elapsed_time(t1), dist, "cuda")
    err_word = st.read_err()

    if not external:  # eager instrumented step: per-launch durations on the launching stream
        with torch.cuda.stream(stream):
            run_step(0, ev_s)
        stream.synchronize()
    # the dominant kernel alone, in the bench's launch configuration: the L decode_layer launches of a step
    # (every unit rescored) back to back in one graph (no event between launches, so programmatic dependent
    # launch still lets each launch's CTAs be scheduled while its predecessor drains); per launch = region /
    # launches
    dl_ms = None
    if path == "decode_layer" and not args.no_graph:
        a = step_inputs(0)
        g_dl = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_dl, stream=stream):
            for l in range(L):
                decode_layer_call(st, l, a["q"][l], a["nk"][l], a["nv"][l], early_reads, None, a.get("tok_begin"),
                                  a.get("seq_len"))
        dl_ms = time_graphs([g_dl], stream, max(3, min(args.steps, 100)))[0] / L
    score_ms = [ev_s[4 * l].elapsed_time(ev_s[4 * l + 1]) for l in range(L)]
    attn_ms = [ev_s[4 * l + 2].elapsed_time(ev_s[4 * l + 3]) for l in range(L)] if path == "unfused" else [0.0]
    peak, peak_kind = peaks()
    sep = None
    if path == "decode_layer" and not episode and not args.no_graph and not args.no_separate_calls:
        sep = separate_calls_leg(st, cfg, L, q_dev, stream, max(3, min(args.steps // 4, 50)), peak)

    # ---- end to end: host buffers in, host results out ------------------------
    # every step copies that step's queries and new K/V rows from pinned host memory, replays its graph, and
    # copies out, lse and the promoted counts to pinned host memory -- overlapped with the compute, as a decode
    # loop runs it: step i+1's inputs cross the link into a staging buffer on a copy stream while step i
    # computes, and step i's results are copied on the device into a staging buffer that a second stream reads
    # back while step i+1 computes.  Two staging sets alternate; events keep each set from being overwritten
    # before it is read.  The on-device copies into the graph's input buffers and out of its outputs run on
    # the compute stream (a few MB each, at HBM rate).
    in_dev = [(a["q"], a["nk"], a["nv"]) for a in (step_inputs(t) for t in range(E))]
    in_host = [tuple(x.cpu().pin_memory() for x in trio) for trio in in_dev]
    out_dev = (st.out, st.lse, st.promoted_cnt)
    out_host = tuple(torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in out_dev)
    in_stage = [tuple(torch.empty_like(x) for x in in_dev[0]) for _ in range(2)]
    out_stage = [tuple(torch.empty_like(x) for x in out_dev) for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in in_host[0])
    d2h = sum(x.numel() * x.element_size() for x in out_host)
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    out_free = [torch.cuda.Event() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 200))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record()
    h2d_stream.wait_stream(stream)  # every copy of the timed region starts after e0
    d2h_stream.wait_stream(stream)
    for i in range(e2e_steps):
        t, b = i % E, i % 2
        with torch.cuda.stream(h2d_stream):  # host -> staging set b, once step i - 2 has taken it
            h2d_stream.wait_event(in_free[b])
            for d, h in zip(in_stage[b], in_host[t]):
                d.copy_(h, non_blocking=True)
            in_ready[b].record()
        with torch.cuda.stream(stream):
            stream.wait_event(in_ready[b])
            for d, sg in zip(in_dev[t], in_stage[b]):
                d.copy_(sg, non_blocking=True)
            in_free[b].record()
            graphs[t].replay()
            stream.wait_event(out_free[b])  # step i - 2's results have left staging set b
            for sg, d in zip(out_stage[b], out_dev):
                sg.copy_(d, non_blocking=True)
            out_ready[b].record()
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(out_ready[b])
            for h, sg in zip(out_host, out_stage[b]):
                h.copy_(sg, non_blocking=True)
            out_free[b].record()
    with torch.cuda.stream(stream):
        stream.wait_stream(d2h_stream)
        e1.record()
    stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    acc_all = algorithmic_bytes(cfg)
    if episode:  # the bytes of the steps actually timed: every unit on a rerank step, else the unstable heads'
        tot = sum(algorithmic_bytes(cfg, rescored_units=ep.rescored_units(t, cfg.B))["total"] for t in timed_steps)
        acc = {"total": tot / len(timed_steps)}
    else:
        acc = acc_all
    n_ls = args.steps * L * world
    secs = ms_total / 1e3
    value = n_ls / secs
    kv_gbs = acc["total"] * n_ls / secs / 1e9
    s_ms, a_ms = statistics.mean(score_ms), statistics.mean(attn_ms)
    if path == "decode_layer":
        dom, dom_ms, dom_bytes = "decode_layer", (dl_ms if dl_ms is not None else s_ms), acc_all["decode_launch"]
        kernel_ms = {"decode_layer": dom_ms, "decode_layer_event_bracketed": s_ms}
    elif path == "fused":
        dom, dom_ms, dom_bytes = "page_score_topk_attn", s_ms, acc_all["fused_launch"]
        kernel_ms = {"page_score_topk_attn": s_ms}
    else:
        dom = "sparse_paged_decode_attn" if a_ms >= s_ms else "page_score_topk"
        dom_ms = max(a_ms, s_ms)
        dom_bytes = acc_all["attn_launch"] if a_ms >= s_ms else acc_all["score_launch"]
        kernel_ms = {"page_score_topk": s_ms, "sparse_paged_decode_attn": a_ms}
    kernel_ms["per_layer_step_ms"] = ms_total / args.steps / L
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    traffic = load_traffic(dom, workloads.CONFIGS[args.config].name, cfg.B)
    clk = clocks.summary()
    step_desc = (f"one decode step = {L} layer-steps, " + ("eager launches" if args.no_graph else "CUDA graph replay"))
    if episode:
        step_desc += (f"; steps cycle through a {E}-step episode (drifting queries, one appended token per step, "
                      f"every unit rescored every {ep.period} steps and the unstable heads' units in between)")
    line = {
        "metric": METRIC, "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate",
        "data": "synthetic (seeded; stands in for Llama-3.1-8B long-context decode)",
        "config": {"workload": cfg.name, "layers": L, "global_batch": cfg.B * world, "seq_len": cfg.S,
                   "q_heads": cfg.Hq, "kv_heads": cfg.Hkv, "head_dim": cfg.D, "page_tokens": cfg.T,
                   "top_k_pages": cfg.K, **launch_shape, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2 ({L * (acc_all['meta'] + acc_all['kv']) / 2**30:.1f} GiB of distinct "
                         "data per step, no flush)",
                   "step": step_desc,
                   "path": {"decode_layer": "decode_layer (append, score, select, attend: one launch)",
                            "fused": "kv_minmax_update + page_score_topk_attn (score, select, attend: one "
                                     "launch)",
                            "unfused": "kv_minmax_update + page_score_topk + sparse_paged_decode_attn"}[path],
                   **({"decode_flags": "KVMM_DECODE_EARLY_READS" if early_reads else 0}
                      if path == "decode_layer" else {})},
        "kv_gbs": kv_gbs, "pct_hbm_peak": kv_gbs / peak,
        "bytes_per_layer_step": acc["total"],
        "kernel_ms": kernel_ms,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "kernel": dom,
                     "peak_source": f"{peak_kind} hbm_gbs (burst copy)",
                     "achieved_bytes_per_launch": dom_bytes, "launch_ms": dom_ms,
                     "launch_timing": (f"CUDA events around {L}-launch graph replays of decode_layer alone "
                                       "(every unit rescored), back to back; per launch = region / launches"
                                       if dl_ms is not None else
                                       "CUDA events around each launch in the last timed step"
                                       if external else "CUDA events, eager instrumented step after timing")},
        "e2e": {"value": e2e_steps * L * world / (e2e_ms / 1e3), "unit": "layer-steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "every step: pinned host q/new K,V -> device (copy stream, overlapping the previous step), "
                       "graph replay, out/lse/promoted counts -> pinned host (second stream, overlapping the next "
                       "step); two staging sets"},
        # per layer: decode_layer, diff; or update, page_score_topk_attn, diff (fused); or update, scoring,
        # attention, diff (unfused).  Where the clustered kernel does not fit the shape, decode_layer falls back
        # to update + the two-kernel fused path, the fused call to a scoring and a selecting attention kernel,
        # and page_score_topk to a scoring and a selection kernel
        "gpu_launches": {"decode_layer": 2 if one_launch else 4, "fused": 3 if clustered else 4,
                         "unfused": 4 if clustered else 5}[path] * L * args.steps,
        "clocks": clk,
        "device_err": err_word,
    }
    if sep is not None:
        line["separate_calls"] = sep
    if promotions is not None:
        line["promotions"] = promotions
    par = load_parity(workloads.CONFIGS[args.config].name, launch_shape, early_reads)
    if par is not None:
        line["parity"] = par
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg)
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def stability_arm(args):
    """Head-stability profiling at the 8B-32K shape (B 8, L 32, Hkv 8, K 128): record one decode step's
    selections of every layer into a W-step ring, then the RCO of every unit over the window and the
    classification.  Timed with CUDA events on the launching stream; latency-bound kernels, reported in us."""
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm
    from paged_kv_cache_minmax_gb300.runtime import StabilityProfiler

    kbuild.build_library()
    kvmm.load()
    cfg, W = CFG, 16
    shape = kvmm.make_shape(cfg.B, cfg.L, cfg.Hq, cfg.Hkv, cfg.D, cfg.T, cfg.Pmax, cfg.K, 1)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(cfg.seed + 17)
    units = cfg.B * cfg.L * cfg.Hkv
    sel = torch.rand(units, cfg.P, generator=gen, device="cuda").topk(cfg.K, dim=1).indices.sort(dim=1).values
    sel_idx = sel.to(torch.int32).view(cfg.B, cfg.L, cfg.Hkv, cfg.K).contiguous()
    sel_cnt = torch.full((cfg.B, cfg.L, cfg.Hkv), cfg.K, dtype=torch.int32, device="cuda")
    seq_len = torch.full((cfg.B,), cfg.S, dtype=torch.int32, device="cuda")

    class _State:
        pass

    state = _State()
    state.sel_idx, state.sel_cnt, state.seq_len = sel_idx, sel_cnt, seq_len
    prof = StabilityProfiler(shape, W)
    for _ in range(W):
        prof.record(state)
    # each call is captured in a CUDA graph and replayed, so the events time the device, not the host
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # the set-up above ran on the default stream
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    reps = max(args.steps, 20)
    with torch.cuda.stream(stream):
        for _ in range(3):
            prof.record(state)
            prof.classify(lag=1)
    stream.synchronize()
    g_rec, g_rco = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_rec, stream=stream):
        prof.record(state)
    with torch.cuda.graph(g_rco, stream=stream):
        prof.classify(lag=1)
    with torch.cuda.stream(stream):
        for _ in range(3):
            g_rec.replay()
            g_rco.replay()
        e[0].record()
        for _ in range(reps):
            g_rec.replay()
        e[1].record()
        for _ in range(reps):
            g_rco.replay()
        e[2].record()
    stream.synchronize()
    rec_us = e[0].elapsed_time(e[1]) * 1e3 / reps
    rco_us = e[1].elapsed_time(e[2]) * 1e3 / reps
    pairs = W - 1
    rco_bytes = (W * units * (cfg.K + 1) * 4 + W * cfg.B * 4) + units * 4 + cfg.L * cfg.Hkv * 5
    print(json.dumps({
        "metric": "head-stability profiling: RCO over a W-step window, 8B-32K shape", "unit": "us",
        "higher_is_better": False, "record_step_us": rec_us, "rco_classify_us": rco_us,
        "config": {"workload": cfg.name, "units": units, "window": W, "pairs_per_unit": pairs, "top_k": cfg.K,
                   "layers": cfg.L},
        "rco_bytes_read": rco_bytes, "rco_gbs": rco_bytes / (rco_us * 1e-6) / 1e9,
        "device_err": int(prof.err.item())}), flush=True)


def promote_arm(args):
    """Promotion transfer at the 8B-32K shape, one layer: every unit (64) brings 38 pages (30% of its top-128,
    within the 23-35% the FlexiCache summary reports per rerank) from a pinned host store into the blocks of
    38 evicted pages.  Calls alternate between two selections so that every call moves the same pages; each
    pair of calls is one CUDA graph replay.  Reported per grid bound: GB/s of K/V moved over the host link."""
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm

    kbuild.build_library()
    kvmm.load()
    cfg = CFG
    B, Hkv, T, D, Pmax, K = cfg.B, cfg.Hkv, cfg.T, cfg.D, cfg.Pmax, cfg.K
    n_move = 38
    units = B * Hkv
    gen = torch.Generator()
    gen.manual_seed(cfg.seed + 23)
    host_k = torch.empty(B, 1, Hkv, Pmax, T, D, dtype=torch.bfloat16).pin_memory()
    host_v = torch.empty(B, 1, Hkv, Pmax, D, T, dtype=torch.bfloat16).pin_memory()
    host_k.view(torch.int16).random_(generator=gen)
    host_v.view(torch.int16).random_(generator=gen)
    n_phys = units * K
    shape = kvmm.make_shape(B, 1, cfg.Hq, Hkv, D, T, Pmax, K, n_phys)
    k_pool = torch.zeros(n_phys, T, D, dtype=torch.bfloat16, device="cuda")
    v_pool = torch.zeros(n_phys, D, T, dtype=torch.bfloat16, device="cuda")
    # selection A: pages [0, K); selection B: the same with the first n_move replaced by [K, K + n_move)
    bt = torch.full((B, 1, Hkv, Pmax), -1, dtype=torch.int32)
    bt[..., :K] = torch.arange(n_phys, dtype=torch.int32).view(B, 1, Hkv, K)
    bt = bt.cuda()
    ab = torch.arange(K, K + n_move, dtype=torch.int32).expand(B, 1, Hkv, n_move)
    ba = torch.arange(0, n_move, dtype=torch.int32).expand(B, 1, Hkv, n_move)
    lists = {}
    for name, t in (("ab", ab), ("ba", ba)):
        full = torch.zeros(B, 1, Hkv, K, dtype=torch.int32)
        full[..., :n_move] = t
        lists[name] = full.cuda()
    cnt = torch.full((B, 1, Hkv), n_move, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moved = torch.zeros(B, 1, Hkv, dtype=torch.int32, device="cuda")
    bytes_per_call = units * n_move * 2 * T * D * 2
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # the set-up above ran on the default stream
    results = {}
    for ctas in (4, 8, 16, 32, 64, 152):
        def pair():
            kvmm.promote_pages(shape, 0, None, lists["ab"], cnt, lists["ba"], cnt, host_k, host_v, k_pool, v_pool,
                               bt, moved=moved, max_ctas=ctas, err=err)
            kvmm.promote_pages(shape, 0, None, lists["ba"], cnt, lists["ab"], cnt, host_k, host_v, k_pool, v_pool,
                               bt, moved=moved, max_ctas=ctas, err=err)
        with torch.cuda.stream(stream):
            for _ in range(3):
                pair()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            pair()
        reps = max(10, min(args.steps, 100))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        stream.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (2 * reps)
        results[str(ctas)] = {"us_per_call": us, "gbs": bytes_per_call / (us * 1e-6) / 1e9}
    ok = int(err.item()) == 0 and int(moved.min()) == n_move

    # baselines of the same bytes: one cudaMemcpyAsync per promoted page's keys and one per its values (into
    # the blocks the kernel uses), and one contiguous copy of that many bytes from pinned memory
    def copies():
        for b in range(B):
            for h in range(Hkv):
                for i in range(n_move):
                    phys = (b * Hkv + h) * K + i
                    k_pool[phys].copy_(host_k[b, 0, h, K + i], non_blocking=True)
                    v_pool[phys].copy_(host_v[b, 0, h, K + i], non_blocking=True)
    big_h = torch.empty(bytes_per_call // 2, dtype=torch.bfloat16).pin_memory()
    big_d = torch.empty(bytes_per_call // 2, dtype=torch.bfloat16, device="cuda")
    baselines = {}
    for name, fn, r in (("memcpy_per_page", copies, 5), ("memcpy_contiguous", lambda: big_d.copy_(big_h, non_blocking=True),
                                                         max(10, min(args.steps, 100)))):
        with torch.cuda.stream(stream):
            fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        us = time_graphs([g], stream, r)[0] * 1e3
        baselines[name] = {"us_per_call": us, "gbs": bytes_per_call / (us * 1e-6) / 1e9}
    print(json.dumps({
        "metric": "promotion transfer: K/V moved from pinned host memory into recycled blocks", "unit": "GB/s",
        "higher_is_better": True, "bytes_per_call": bytes_per_call, "by_max_ctas": results,
        "baselines": baselines,
        "config": {"workload": cfg.name, "units": units, "pages_per_unit": n_move, "top_k": K,
                   "page_bytes_kv": 2 * T * D * 2, "host_store": "pinned (cudaHostAlloc through torch)"},
        "device_err": int(err.item()), "all_moved": ok}), flush=True)


def table_update_arm(args):
    """Dirty-tracked block-table synchronisation at the 8B-32K shape: one rerank of every unit of every layer
    changes 76 entries per unit (38 promoted pages take blocks, 38 evicted pages become null), 155,648 entries
    of the 4 Mi-entry table.  Timed: block_table_update reading those entries from pinned host memory, against
    copying the whole table from pinned host memory; each as a CUDA graph replay."""
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm

    kbuild.build_library()
    kvmm.load()
    cfg = CFG
    B, L, Hkv, Pmax = cfg.B, cfg.L, cfg.Hkv, cfg.Pmax
    units = B * L * Hkv
    n_phys = units * cfg.K
    shape = kvmm.make_shape(B, L, cfg.Hq, Hkv, cfg.D, cfg.T, Pmax, cfg.K, n_phys)
    gen = torch.Generator()
    gen.manual_seed(cfg.seed + 29)
    table = torch.full((B, L, Hkv, Pmax), -1, dtype=torch.int32, device="cuda")
    host_table = torch.empty(B, L, Hkv, Pmax, dtype=torch.int32).pin_memory()
    host_table.copy_(table.cpu())
    per_unit = 76
    cols = torch.stack([torch.randperm(Pmax, generator=gen)[:per_unit] for _ in range(units)])  # [units, 76]
    idx = (torch.arange(units, dtype=torch.int64)[:, None] * Pmax + cols).reshape(-1).contiguous().pin_memory()
    val = torch.randint(-1, n_phys, (idx.numel(),), generator=gen, dtype=torch.int32).pin_memory()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # the set-up above ran on the default stream

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    reps = max(10, min(args.steps, 200))
    delta_us = timed(lambda: kvmm.block_table_update(shape, idx, val, table, err=err), reps)
    full_us = timed(lambda: table.copy_(host_table, non_blocking=True), reps)
    print(json.dumps({
        "metric": "block-table synchronisation per rerank step: changed entries vs the whole table", "unit": "us",
        "higher_is_better": False, "delta_us": delta_us, "full_table_copy_us": full_us,
        "delta_bytes": idx.numel() * 12, "table_bytes": table.numel() * 4, "changed_entries": idx.numel(),
        "config": {"workload": cfg.name, "units": units, "changed_per_unit": per_unit,
                   "deltas": "pinned host memory, read by the kernel"},
        "device_err": int(err.item())}), flush=True)


def meankey_arm(args):
    """KVDrive's mean-key scorer beside MinMax at the 8B-32K shape (one layer, 64 units, K = 128): the time of
    scoring + top-K for each (CUDA-graph replays; the mean rows are half the bytes), and, over a sample of units,
    the dense attention mass their selections capture (oracle, fp64), next to the best possible: the K pages of
    most mass."""
    import oracle
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm
    from paged_kv_cache_minmax_gb300.runtime import DecodeState
    from paged_kv_cache_minmax_gb300.workloads import bf16_bits

    kbuild.build_library()
    kvmm.load()
    oracle.build()
    cfg = workloads.scaled(CFG, L=1)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    shape = st.shape
    mean = torch.zeros(cfg.B, 1, cfg.Hkv, cfg.Pmax, cfg.D, dtype=torch.bfloat16, device="cuda")
    kvmm.kv_meankey_update(shape, 0, None, wl.seq_len, wl.k_pool, wl.block_table, mean, err=st.err)
    sel_mm = torch.zeros_like(st.sel_idx)
    cnt_mm = torch.zeros_like(st.sel_cnt)
    sel_mk = torch.zeros_like(st.sel_idx)
    cnt_mk = torch.zeros_like(st.sel_cnt)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # the set-up above ran on the default stream

    def timed(fn, reps):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            e0.record()
            for _ in range(reps):
                g.replay()
            e1.record()
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / reps

    reps = max(10, min(args.steps, 200))
    mm_us = timed(lambda: kvmm.page_score_topk(shape, 0, wl.q[0], st.meta, wl.seq_len, None, cfg.K, sel_mm, cnt_mm,
                                               st.workspace, st.err), reps)
    mk_us = timed(lambda: kvmm.page_score_topk_mean(shape, 0, wl.q[0], mean, wl.seq_len, None, cfg.K, sel_mk,
                                                    cnt_mk, st.workspace, st.err), reps)
    torch.cuda.synchronize()
    kp, qb = bf16_bits(wl.k_pool).reshape(-1, cfg.T, cfg.D), bf16_bits(wl.q[0])
    captured = {"minmax": [], "meankey": [], "best": []}
    sample = [(b, h) for b in range(cfg.B) for h in range(0, cfg.Hkv, 4)][:max(2, min(16, args.steps))]
    for b, h in sample:
        row = wl.block_table[b, 0, h].cpu().numpy()
        seq = int(wl.seq_len[b])
        mass = oracle.unit_page_mass(qb[b, h * cfg.G:(h + 1) * cfg.G], kp, cfg.T, row, seq).mean(axis=0)
        for name, sel, cnt in (("minmax", sel_mm, cnt_mm), ("meankey", sel_mk, cnt_mk)):
            pages = sel[b, 0, h, :int(cnt[b, 0, h])].cpu().numpy()
            captured[name].append(float(mass[pages].sum()))
        captured["best"].append(float(np.sort(mass)[::-1][:cfg.K].sum()))
    meta_bytes = cfg.B * cfg.Hkv * cfg.P * 2 * cfg.D * 2
    print(json.dumps({
        "metric": "page scorers: MinMax bounds vs mean key (KVDrive); time and dense attention mass captured",
        "unit": "us", "higher_is_better": False,
        "score_topk_us": {"minmax": mm_us, "meankey": mk_us},
        "metadata_bytes": {"minmax": meta_bytes, "meankey": meta_bytes // 2},
        "attention_mass_captured_mean": {k: float(np.mean(v)) for k, v in captured.items()},
        "attention_mass_captured_min": {k: float(np.min(v)) for k, v in captured.items()},
        "config": {"workload": cfg.name, "units": cfg.B * cfg.Hkv, "top_k": cfg.K, "pages": cfg.P,
                   "sampled_units": len(sample), "keys": cfg.key_dist, "planted_pages": cfg.n_planted},
        "device_err": st.read_err()}), flush=True)


def centroid_arm(args):
    """KVDrive's centroid level at the 8B-32K shape (one layer, 64 units, K = 128): the index build and the
    two-level selection for a spatial blocking (R = 4 pages a centroid, no iteration) and for the k-means
    grouping with half the centroids (R = 8, 3 Lloyd iterations), each expanding M = 4K / R centroids (about
    4K pages); beside MinMax and the flat mean-key scorer.  Times are CUDA-graph replays; over a sample of
    units, the dense attention mass each selection captures (oracle, fp64), next to the best possible: the K
    pages of most mass."""
    import oracle
    from paged_kv_cache_minmax_gb300 import build as kbuild
    from paged_kv_cache_minmax_gb300 import kvmm
    from paged_kv_cache_minmax_gb300.runtime import DecodeState
    from paged_kv_cache_minmax_gb300.workloads import bf16_bits

    kbuild.build_library()
    kvmm.load()
    oracle.build()
    cfg = workloads.scaled(CFG, L=1)
    wl = workloads.generate(cfg, device="cuda")
    st = DecodeState.for_workload(wl)
    st.build_metadata()
    shape = st.shape
    mean = torch.zeros(cfg.B, 1, cfg.Hkv, cfg.Pmax, cfg.D, dtype=torch.bfloat16, device="cuda")
    kvmm.kv_meankey_update(shape, 0, None, wl.seq_len, wl.k_pool, wl.block_table, mean, err=st.err)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    reps = max(10, min(args.steps, 200))

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return time_graphs([g], stream, reps)[0] * 1e3

    sels = {}
    times = {}

    def new_sel():
        return torch.zeros_like(st.sel_idx), torch.zeros_like(st.sel_cnt)

    sels["minmax"] = new_sel()
    times["minmax_score_topk_us"] = timed(lambda: kvmm.page_score_topk(
        shape, 0, wl.q[0], st.meta, wl.seq_len, None, cfg.K, *sels["minmax"], st.workspace, st.err))
    sels["meankey"] = new_sel()
    times["meankey_score_topk_us"] = timed(lambda: kvmm.page_score_topk_mean(
        shape, 0, wl.q[0], mean, wl.seq_len, None, cfg.K, *sels["meankey"], st.workspace, st.err))
    variants = {"spatial_r4": (4, 0), "kmeans_r8_it3": (8, 3)}
    index_bytes = {}
    for name, (R, n_iter) in variants.items():
        cmax = kvmm.centroid_rows(shape, R)
        cent = torch.zeros(cfg.B, 1, cfg.Hkv, cmax, cfg.D, dtype=torch.bfloat16, device="cuda")
        assign = torch.zeros(cfg.B, 1, cfg.Hkv, cfg.Pmax, dtype=torch.int32, device="cuda")
        off = torch.zeros(cfg.B, 1, cfg.Hkv, cmax + 1, dtype=torch.int32, device="cuda")
        members = torch.zeros_like(assign)
        times[name + "_build_us"] = timed(lambda: kvmm.kv_centroid_build(
            shape, 0, mean, wl.seq_len, R, n_iter, cent, assign, off, members, err=st.err))
        sels[name] = new_sel()
        M = max(1, 4 * cfg.K // R)
        times[name + "_select_us"] = timed(lambda: kvmm.page_score_topk_centroid(
            shape, 0, wl.q[0], mean, wl.seq_len, R, cent, off, members, None, M, cfg.K, *sels[name], err=st.err))
        index_bytes[name] = {"centroids": cfg.B * cfg.Hkv * ((cfg.P + R - 1) // R) * cfg.D * 2, "M": M,
                             "pages_expanded": M * R}
    torch.cuda.synchronize()
    kp, qb = bf16_bits(wl.k_pool).reshape(-1, cfg.T, cfg.D), bf16_bits(wl.q[0])
    captured = {k: [] for k in list(sels) + ["best"]}
    sample = [(b, h) for b in range(cfg.B) for h in range(0, cfg.Hkv, 4)][:max(2, min(16, args.steps))]
    for b, h in sample:
        row = wl.block_table[b, 0, h].cpu().numpy()
        seq = int(wl.seq_len[b])
        mass = oracle.unit_page_mass(qb[b, h * cfg.G:(h + 1) * cfg.G], kp, cfg.T, row, seq).mean(axis=0)
        for name, (sel, cnt) in sels.items():
            pages = sel[b, 0, h, :int(cnt[b, 0, h])].cpu().numpy()
            captured[name].append(float(mass[pages].sum()))
        captured["best"].append(float(np.sort(mass)[::-1][:cfg.K].sum()))
    print(json.dumps({
        "metric": "KVDrive centroid index: build and two-level selection time; dense attention mass captured",
        "unit": "us", "higher_is_better": False, "times_us": times, "index": index_bytes,
        "attention_mass_captured_mean": {k: float(np.mean(v)) for k, v in captured.items()},
        "attention_mass_captured_min": {k: float(np.min(v)) for k, v in captured.items()},
        "config": {"workload": cfg.name, "units": cfg.B * cfg.Hkv, "top_k": cfg.K, "pages": cfg.P,
                   "sampled_units": len(sample), "keys": cfg.key_dist, "planted_pages": cfg.n_planted},
        "device_err": st.read_err()}), flush=True)


def load_parity(workload, launch_shape, early_reads):
    """The GPU-versus-oracle parity record of ``workload`` at the benchmark's launch shape, written by the
    ``-m gpu`` tests (tests/test_gpu_bench_shapes.py) into profiles/parity.json, with two checks: whether it
    was taken with the current CUDA sources, and whether its launch shape and flags are the ones timed here."""
    from paged_kv_cache_minmax_gb300 import build as kbuild

    path = os.path.join(ROOT, "profiles", "parity.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if rec is None:
        return None
    out = dict(rec)
    out["current_sources"] = rec.get("sources") == kbuild.source_digest()
    mine = {k: launch_shape[k] for k in ("units_per_cluster", "cluster_ctas") if k in launch_shape}
    out["launch_shape_matches"] = (rec.get("launch_shape") == mine and
                                   bool(rec.get("early_reads")) == bool(early_reads))
    return out


def load_traffic(kernel, workload, batch):
    """dram bytes per launch of ``kernel`` on ``workload`` from the committed ncu summaries, if one was
    captured at that batch (a launch covers one layer, so the layer count does not matter) with the current
    CUDA sources: a capture of an earlier kernel no longer describes this one."""
    from paged_kv_cache_minmax_gb300 import build as kbuild

    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(kernel, {}).get(workload)
    if not rec or rec["batch"] != batch or rec.get("sources") != kbuild.source_digest():
        return None
    return rec["bytes"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="kvmm", choices=["kvmm", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--config", type=int, default=2, choices=sorted(workloads.CONFIGS),
                    help="workload (default: the 8B-shape 32K-context decode step)")
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly (for profilers)")
    ap.add_argument("--clocks-log", default=None,
                    help="also write the nvidia-smi clock samples of the timed region to this CSV file")
    ap.add_argument("--batch", type=int, default=0, help="override the batch (smaller profiling case)")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (smaller profiling case)")
    ap.add_argument("--meankey", action="store_true",
                    help="compare the mean-key scorer with MinMax (time, attention mass captured) instead")
    ap.add_argument("--centroid", action="store_true",
                    help="time KVDrive's centroid index (build, two-level selection) and compare attention mass")
    ap.add_argument("--table-update", action="store_true",
                    help="time dirty-tracked block-table synchronisation instead")
    ap.add_argument("--promote", action="store_true",
                    help="time the promotion transfer from pinned host memory instead")
    ap.add_argument("--stability", action="store_true",
                    help="time head-stability profiling (history record, RCO and classification) instead")
    ap.add_argument("--no-separate-calls", action="store_true",
                    help="skip timing page_score_topk and sparse_paged_decode_attn as separate calls")
    ap.add_argument("--no-early-reads", action="store_true",
                    help="decode_layer waits for the preceding kernel before any read (no KVMM_DECODE_EARLY_READS)")
    ap.add_argument("--path", default="decode_layer", choices=["decode_layer", "fused", "unfused"],
                    help="decode_layer (one launch per layer), fused (kv_minmax_update + page_score_topk_attn) "
                         "or unfused (kv_minmax_update + page_score_topk + sparse_paged_decode_attn)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        reference_arm(args)
    elif args.stability:
        stability_arm(args)
    elif args.promote:
        promote_arm(args)
    elif args.table_update:
        table_update_arm(args)
    elif args.meankey:
        meankey_arm(args)
    elif args.centroid:
        centroid_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
