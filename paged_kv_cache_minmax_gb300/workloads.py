"""Seeded synthetic inputs shaped like long-context GQA decode workloads.

This module creates inputs only: queries, key/value pools, head-level block
tables, sequence lengths, appended tokens and the stable/unstable head split.
It holds none of the method's arithmetic (no MinMax, scoring, selection or
attention), so both the CUDA path and the CPU oracle may consume what it
makes.  The pages evaluate on trained models and datasets (Llama-3.1-8B,
L-Eval, LongBench) that are not available here; these generators stand in for
their shapes.

Recipe (every tensor is drawn from one ``torch.Generator`` seeded per config):
  * V ~ N(0, 1) in bf16.
  * K ~ N(0, 1) in bf16, then per (layer, KV head):
      - "normal":    unchanged;
      - "outlier":   4 seeded channels multiplied by 8;
      - "chanscale": every channel multiplied by a seeded factor in U[0.5, 4].
  * planted pages: per unit, ``n_planted`` distinct seeded logical pages get
    k <- bf16(k + beta * u) on every token, u = (sum of the group's query
    heads) / its 2-norm, beta = 4, so the top-K set is not arbitrary.
  * q ~ N(0, 1) in bf16 per layer; with drift, q_t = 0.9 q_{t-1} + 0.44 eps
    in fp32 (eps ~ N(0, 1)), rounded to bf16 for use.
  * physical pool: identity layout (unit-major, logical page order) or a
    seeded random permutation of the physical pages; K pages are stored
    token by token ([T][D]), V pages dimension by dimension ([D][T]).
  * stable/unstable split: a seeded subset of ``unstable_frac`` of the
    (layer, KV head) pairs is unstable.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Config:
    """One workload shape. ``S`` counts tokens including the current one."""

    name: str
    B: int
    L: int
    Hq: int
    Hkv: int
    D: int
    T: int
    S: int
    K: int
    key_dist: str = "normal"  # "normal" | "outlier" | "chanscale"
    n_planted: int = 0
    permuted_pool: bool = False
    steps: int = 0  # decode steps that append one token each
    unstable_frac: float = 0.0
    rerank_period: int = 16
    beta: float = 4.0
    seed: int = 1000
    ragged: bool = False  # per-batch sequence lengths S - b*(T+3) (ragged tails)
    layers_alloc: int | None = None  # allocate only this many layers (rotated)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def P(self) -> int:
        return -(-self.S // self.T)

    @property
    def Pmax(self) -> int:
        return -(-(self.S + self.steps) // self.T)

    @property
    def L_alloc(self) -> int:
        return min(self.layers_alloc, self.L) if self.layers_alloc else self.L

    def seq_lens(self) -> list[int]:
        if not self.ragged:
            return [self.S] * self.B
        return [max(1, self.S - b * (self.T + 3)) for b in range(self.B)]


CONFIGS: dict[int, Config] = {
    1: Config("tiny-b1-h4x1-d64-t16-s1024-k8", B=1, L=1, Hq=4, Hkv=1, D=64, T=16, S=1024, K=8,
              seed=1001),
    2: Config("llama8b-32k-b8-k128", B=8, L=32, Hq=32, Hkv=8, D=128, T=16, S=32768, K=128,
              key_dist="outlier", n_planted=128, seed=1002),
    3: Config("llama8b-128k-b4-k256-permuted", B=4, L=32, Hq=32, Hkv=8, D=128, T=16, S=131072, K=256,
              key_dist="outlier", n_planted=128, permuted_pool=True, seed=1003),
    4: Config("llama8b-16k-b32-k128-mix25", B=32, L=32, Hq=32, Hkv=8, D=128, T=16, S=16384, K=128,
              key_dist="outlier", n_planted=128, steps=64, unstable_frac=0.25, seed=1004),
    5: Config("gqa5-64k-b16-t32-k64", B=16, L=64, Hq=40, Hkv=8, D=128, T=32, S=65536, K=64,
              key_dist="chanscale", n_planted=128, seed=1005, layers_alloc=8),
}


def scaled(cfg: Config, **kw) -> Config:
    """A smaller copy of ``cfg`` (for parity runs the oracle finishes in seconds)."""
    return replace(cfg, **kw)


@dataclass
class Workload:
    cfg: Config
    q: torch.Tensor  # [L_alloc, B, Hq, D] bf16
    k_pool: torch.Tensor  # [Nphys, T, D] bf16 (token-major pages)
    v_pool: torch.Tensor  # [Nphys, D, T] bf16 (dimension-major pages)
    block_table: torch.Tensor  # [B, L_alloc, Hkv, Pmax] int32
    seq_len: torch.Tensor  # [B] int32
    unstable: torch.Tensor  # [L_alloc, Hkv] uint8
    key_scale: torch.Tensor  # [L_alloc, Hkv, D] float32 (channel factors used for K)
    planted: torch.Tensor  # [B, L_alloc, Hkv, n_planted] int64 logical pages (or empty)
    extra: dict = field(default_factory=dict)

    @property
    def n_phys(self) -> int:
        return self.k_pool.shape[0]


def _key_scale(cfg: Config, gen: torch.Generator, device) -> torch.Tensor:
    L, H, D = cfg.L_alloc, cfg.Hkv, cfg.D
    scale = torch.ones(L, H, D, dtype=torch.float32, device=device)
    if cfg.key_dist == "outlier":
        for l in range(L):
            for h in range(H):
                ch = torch.randperm(D, generator=gen, device=device)[:4]
                scale[l, h, ch] = 8.0
    elif cfg.key_dist == "chanscale":
        scale = 0.5 + 3.5 * torch.rand(L, H, D, generator=gen, device=device)
    return scale


def _scale_keys(k: torch.Tensor, scale_rows: torch.Tensor) -> None:
    """k [n, T, D] bf16 *= scale_rows [n, D] (rounded to bf16), in place."""
    k.copy_((k.float() * scale_rows[:, None, :]).to(torch.bfloat16))


def generate(cfg: Config, device="cpu", seed: int | None = None, chunk_pages: int = 1 << 17) -> Workload:
    """Build the full seeded workload of ``cfg`` on ``device``."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed if seed is None else seed)
    B, L, Hq, Hkv, D, T, Pmax = cfg.B, cfg.L_alloc, cfg.Hq, cfg.Hkv, cfg.D, cfg.T, cfg.Pmax
    n_units = B * L * Hkv
    n_phys = n_units * Pmax

    q = torch.randn(L, B, Hq, D, generator=gen, device=device).to(torch.bfloat16)
    key_scale = _key_scale(cfg, gen, device)

    if cfg.permuted_pool:
        perm = torch.randperm(n_phys, generator=gen, device=device)
        block_table = perm.to(torch.int32).view(B, L, Hkv, Pmax)
    else:
        block_table = torch.arange(n_phys, device=device, dtype=torch.int32).view(B, L, Hkv, Pmax)

    # (layer, head) of every physical page, through the table
    unit_lh = (torch.arange(L, device=device)[:, None] * Hkv + torch.arange(Hkv, device=device)[None, :])
    lh_logical = unit_lh[None, :, :, None].expand(B, L, Hkv, Pmax).reshape(-1)
    lh_of_phys = torch.empty(n_phys, dtype=torch.int64, device=device)
    lh_of_phys[block_table.reshape(-1).long()] = lh_logical

    k_pool = torch.empty(n_phys, T, D, dtype=torch.bfloat16, device=device)
    v_pool = torch.empty(n_phys, D, T, dtype=torch.bfloat16, device=device)
    flat_scale = key_scale.view(L * Hkv, D)
    for s in range(0, n_phys, chunk_pages):
        e = min(n_phys, s + chunk_pages)
        k_pool[s:e] = torch.randn(e - s, T, D, generator=gen, device=device).to(torch.bfloat16)
        v_pool[s:e] = torch.randn(e - s, D, T, generator=gen, device=device).to(torch.bfloat16)
        if cfg.key_dist != "normal":
            _scale_keys(k_pool[s:e], flat_scale[lh_of_phys[s:e]])

    seq_len = torch.tensor(cfg.seq_lens(), dtype=torch.int32, device=device)

    planted = torch.empty(B, L, Hkv, 0, dtype=torch.int64, device=device)
    if cfg.n_planted > 0:
        n_pl = min(cfg.n_planted, cfg.P)
        keys = torch.rand(B, L, Hkv, cfg.P, generator=gen, device=device)
        planted = keys.argsort(dim=-1)[..., :n_pl]
        # direction: normalised sum of the group's query heads, per (l, b, kv head)
        qg = q.float().view(L, B, Hkv, cfg.G, D).sum(dim=3)
        u = qg / qg.norm(dim=-1, keepdim=True)
        u = u.permute(1, 0, 2, 3)  # [B, L, Hkv, D]
        phys = torch.gather(block_table.long(), 3, planted)  # [B, L, Hkv, n_pl]
        shift = (cfg.beta * u)[:, :, :, None, None, :]  # [B,L,Hkv,1,1,D]
        for b in range(B):
            idx = phys[b].reshape(-1)
            pages = k_pool[idx].float().view(L, Hkv, n_pl, T, D)
            pages += shift[b].view(L, Hkv, 1, 1, D)
            k_pool[idx] = pages.view(-1, T, D).to(torch.bfloat16)

    unstable = torch.zeros(L, Hkv, dtype=torch.uint8, device=device)
    if cfg.unstable_frac > 0:
        n_unst = int(round(cfg.unstable_frac * L * Hkv))
        pick = torch.randperm(L * Hkv, generator=gen, device=device)[:n_unst]
        unstable.view(-1)[pick] = 1

    return Workload(cfg, q, k_pool, v_pool, block_table, seq_len, unstable, key_scale, planted)


def step_tokens(wl: Workload, step: int, device=None) -> tuple[torch.Tensor, torch.Tensor]:
    """New K/V rows ``[L_alloc, B, Hkv, 1, D]`` (bf16) appended at decode step ``step``.

    K follows the same per-(layer, head) channel law as the pool; V ~ N(0,1).
    """
    cfg = wl.cfg
    device = wl.k_pool.device if device is None else device
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 1_000_003 + 7919 * (step + 1))
    L, B, H, D = cfg.L_alloc, cfg.B, cfg.Hkv, cfg.D
    k = torch.randn(L, B, H, 1, D, generator=gen, device=device)
    v = torch.randn(L, B, H, 1, D, generator=gen, device=device)
    k = k * wl.key_scale.to(device)[:, None, :, None, :]
    return k.to(torch.bfloat16), v.to(torch.bfloat16)


def drift_queries(wl: Workload, steps: int) -> torch.Tensor:
    """Queries ``[steps, L_alloc, B, Hq, D]`` (bf16): q_t = 0.9 q_{t-1} + 0.44 eps_t in fp32.

    q_0 is the workload's q.
    """
    cfg = wl.cfg
    device = wl.q.device
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 7 + 3)
    out = torch.empty((steps,) + tuple(wl.q.shape), dtype=torch.bfloat16, device=device)
    state = wl.q.float()
    for t in range(steps):
        if t > 0:
            eps = torch.randn(state.shape, generator=gen, device=device)
            state = 0.9 * state + 0.44 * eps
        out[t] = state.to(torch.bfloat16)
    return out


def drift_queries_by_stability(wl: Workload, steps: int, keep_stable: float = 0.99,
                               keep_unstable: float = 0.3) -> torch.Tensor:
    """Queries ``[steps, L_alloc, B, Hq, D]`` (bf16) whose drift depends on the seeded stable/unstable split:
    q_t = a q_{t-1} + sqrt(1 - a^2) eps_t (fp32; same stationary scale), with a = keep_unstable for the query
    heads of an unstable (layer, KV head) and keep_stable otherwise.  q_0 is the workload's q."""
    cfg = wl.cfg
    device = wl.q.device
    gen = torch.Generator(device=device)
    gen.manual_seed(cfg.seed * 7 + 5)
    unst = wl.unstable.bool().repeat_interleave(cfg.G, dim=1)  # [L_alloc, Hq]
    a = torch.where(unst, torch.tensor(keep_unstable, device=device), torch.tensor(keep_stable, device=device))
    a = a[:, None, :, None]  # [L, 1, Hq, 1]
    out = torch.empty((steps,) + tuple(wl.q.shape), dtype=torch.bfloat16, device=device)
    state = wl.q.float()
    scale = state.std()
    for t in range(steps):
        if t > 0:
            eps = torch.randn(state.shape, generator=gen, device=device) * scale
            state = a * state + torch.sqrt(1 - a * a) * eps
        out[t] = state.to(torch.bfloat16)
    return out


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a (CPU or CUDA) tensor as a numpy uint16 array."""
    import numpy as np

    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def kv_bytes_per_token(L: int, Hkv: int, D: int, elem_bytes: int = 2) -> int:
    """K and V bytes one token occupies across all layers (2 * L * Hkv * D * elem)."""
    return 2 * L * Hkv * D * elem_bytes


def planted_count(cfg: Config) -> int:
    return min(cfg.n_planted, cfg.P) if cfg.n_planted else 0


def describe(cfg: Config) -> str:
    return (f"{cfg.name}: B={cfg.B} L={cfg.L} (alloc {cfg.L_alloc}) Hq={cfg.Hq} Hkv={cfg.Hkv} D={cfg.D} "
            f"T={cfg.T} S={cfg.S} P={cfg.P} K={cfg.K} keys={cfg.key_dist} planted={cfg.n_planted} "
            f"permuted={cfg.permuted_pool} steps={cfg.steps} unstable={cfg.unstable_frac} seed={cfg.seed}")

