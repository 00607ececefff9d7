"""Seeded synthetic inputs for decode-phase hybrid sparse attention.

This module only draws random numbers and lays them out in the paged-KV
format; it holds none of the attention / selection arithmetic.  Both the CUDA
path (through the C-ABI binding) and the fp64 oracle consume what it returns.

Recipe (the value distributions are a reading of the workloads the pages
describe; no public dataset is reproduced):

* Q, K, V entries are N(0, 1).  The softmax scale is 1/sqrt(D).  (The
  "scaled 1/sqrt(128)" in the workload text is read as the softmax scale.)
* GQA realism: inside a KV-head group, q_h = sqrt(.5) z_g + sqrt(.5) z_h with
  z_g shared by the group.  The group direction is
  g_hat = normalise(mean_h q_h) * sqrt(D).
* Attention sink: key 0 of every (sequence, KV head) gets + c_sink * g_hat.
  The sink phenomenon is the one the Fluxion page measures (Fig. 3c, Fig. 4).
* Heavy blocks: a set of candidate blocks (block size of that KV head) whose
  every key gets + c_heavy * g_hat.
* Recency bias (optional): key t in the last R tokens gets + ramp(t) * g_hat,
  ramp rising linearly from 0 to 1 (HGCA: recent entries dominate attention).
* The page table is a seeded random permutation of physical pages, so the
  gather through it is a real scatter over the pool.
* Sink-dominated heads (optional, the sparsity-bypass workloads): in each
  sequence `sink_heads` query heads, drawn at random, get
  q_h += c_qsink * k_0 / |k_0| with k_0 their KV head's key 0, so their
  attention is held by the first token (LFPS measures about 12 % of heads
  bypassed at epsilon = 0.85).

Draw order (fixed, so a seed reproduces a case): group noise z_g, head noise
z_h, K pool, V pool, page permutation, heavy-block picks, sink-head picks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

HEAD_DIM = 128
PAGE_SIZE = 16


@dataclass
class Workload:
    """One decode-attention workload: shapes, selection settings, planted structure."""

    name: str
    B: int
    Hq: int
    Hk: int
    L: int                          # tokens in the cache, current token included
    block_sizes: List[int]          # per KV head, each in {8, 16, 32, 64}
    budget_bp: List[int]            # per KV head, budget in basis points of candidate blocks
    S: int = 4                      # attention-sink tokens
    W: int = 1024                   # recent window
    D: int = HEAD_DIM
    P: int = PAGE_SIZE
    mode: str = "minmax"            # block summary kind: "minmax" or "mean"
    c_sink: float = 2.0
    c_heavy: float = 1.5
    heavy_count: Optional[int] = None    # fixed number of heavy blocks per (b, kv head)
    heavy_frac: float = 0.01             # else this fraction of candidate blocks
    recency: int = 0                     # length of the recency ramp (0 = none)
    extra_tokens: int = 0                # page-table room for appended tokens
    lens: Optional[List[int]] = None     # per-sequence lengths (ragged batch); default all L
    sink_heads: int = 0                  # query heads per sequence aligned with key 0
    c_qsink: float = 24.0

    @property
    def G(self) -> int:
        return self.Hq // self.Hk

    @property
    def max_pages_per_seq(self) -> int:
        return (self.L + self.extra_tokens + self.P - 1) // self.P


def _draw_block_settings(Hk: int, seed: int):
    g = torch.Generator().manual_seed(10_000 + seed)
    sizes = [8, 16, 32, 64]
    bs = [sizes[int(torch.randint(0, 4, (1,), generator=g))] for _ in range(Hk)]
    bp = [int(torch.randint(200, 2001, (1,), generator=g)) for _ in range(Hk)]
    return bs, bp


def workload(name: str) -> Workload:
    """The named workloads.  Shapes follow the Llama-3.1-8B / Qwen2.5-7B
    attention layers and the 32K / 5 % budget / batch-8 setting of the Fluxion
    time breakdown (Fig. 2)."""
    if name == "tiny_4k":
        return Workload(name, B=1, Hq=8, Hk=2, L=4096, block_sizes=[16, 16],
                        budget_bp=[1000, 1000], S=4, W=256, c_heavy=2.0, heavy_count=3)
    if name == "llama_32k":
        return Workload(name, B=8, Hq=32, Hk=8, L=32768, block_sizes=[16] * 8,
                        budget_bp=[500] * 8, S=4, W=1024, c_heavy=1.5,
                        heavy_frac=0.01, recency=2048)
    if name == "qwen_64k":
        bs, bp = _draw_block_settings(4, 2)
        return Workload(name, B=16, Hq=28, Hk=4, L=65536, block_sizes=bs,
                        budget_bp=bp, S=4, W=1024, c_heavy=1.5, heavy_frac=0.01,
                        recency=2048)
    if name == "tiny_4k_sinkheads":
        # ragged: a long sequence, a short one, one with no global tokens, one token
        return Workload(name, B=4, Hq=8, Hk=2, L=4096, block_sizes=[16, 16], budget_bp=[1000, 1000], S=4,
                        W=256, c_sink=0.0, c_heavy=2.0, heavy_count=3, lens=[4096, 1000, 7, 1], sink_heads=2)
    if name == "llama_32k_sinkheads":
        return Workload(name, B=8, Hq=32, Hk=8, L=32768, block_sizes=[16] * 8, budget_bp=[500] * 8, S=4,
                        W=1024, c_sink=0.0, c_heavy=1.5, heavy_frac=0.01, recency=2048, sink_heads=4)
    raise KeyError(name)


def sweep_workload(B: int, ctx: int, budget_bp: int, extra_tokens: int = 16) -> Workload:
    """One cell of the throughput sweep of the full decode-attention stack:
    a Llama-3-8B-shaped layer (32 q / 8 KV heads, page = block = 16, 4 sinks,
    window 1024), batch B, context ctx, budget budget_bp basis points of the
    candidate blocks (10000 = dense), room for extra_tokens appended tokens;
    planted sink, 1 % heavy blocks and the 2K recency ramp of the 32K layer."""
    return Workload(f"sweep_b{B}_ctx{ctx}_bp{budget_bp}", B=B, Hq=32, Hk=8, L=ctx, block_sizes=[16] * 8,
                    budget_bp=[budget_bp] * 8, S=4, W=1024, c_heavy=1.5, heavy_frac=0.01, recency=2048,
                    extra_tokens=extra_tokens)


# --------------------------------------------------------------------------
# partition helpers (pure integer bookkeeping, shared by the harness)
# --------------------------------------------------------------------------

def candidate_range(L: int, S: int, W: int, Bs: int):
    """Block index range [j0, j1) of blocks that intersect the middle region
    M = [min(S, L), max(L - W, min(S, L)))."""
    s_end = min(S, L)
    w_beg = max(L - W, s_end)
    if w_beg <= s_end:
        return 0, 0
    return s_end // Bs, (w_beg + Bs - 1) // Bs


def budget_k(bp: int, ncand: int) -> int:
    """k = ceil(bp / 10000 * ncand) in exact integer arithmetic."""
    return min(ncand, (bp * ncand + 9999) // 10000)


def k_per_qhead(wl: Workload, L: Optional[int] = None) -> List[int]:
    L = wl.L if L is None else L
    ks = []
    for h in range(wl.Hq):
        kvh = h // wl.G
        j0, j1 = candidate_range(L, wl.S, wl.W, wl.block_sizes[kvh])
        ks.append(budget_k(wl.budget_bp[kvh], j1 - j0))
    return ks


# --------------------------------------------------------------------------
# the generator
# --------------------------------------------------------------------------

@dataclass
class DecodeCase:
    wl: Workload
    q: torch.Tensor            # bf16 [B, Hq, D]
    k_pool: torch.Tensor       # bf16 [num_pages, Hk, P, D]
    v_pool: torch.Tensor       # bf16 [num_pages, Hk, P, D]
    page_table: torch.Tensor   # int32 [B, max_pages_per_seq]
    seq_lens: torch.Tensor     # int32 [B]
    g_hat: torch.Tensor        # float32 [B, Hk, D]
    heavy: List[List[List[int]]] = field(default_factory=list)  # [b][kvh] -> block ids


def make_decode_case(wl: Workload, seed: int, device="cpu") -> DecodeCase:
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    B, Hq, Hk, G, D, P = wl.B, wl.Hq, wl.Hk, wl.G, wl.D, wl.P
    f32 = torch.float32

    z_g = torch.randn(B, Hk, 1, D, generator=g, device=dev, dtype=f32)
    z_h = torch.randn(B, Hk, G, D, generator=g, device=dev, dtype=f32)
    q = math.sqrt(0.5) * z_g + math.sqrt(0.5) * z_h              # [B, Hk, G, D]
    mean_q = q.mean(dim=2)                                        # [B, Hk, D]
    g_hat = mean_q / mean_q.norm(dim=-1, keepdim=True) * math.sqrt(D)
    q_bf = q.reshape(B, Hq, D).to(torch.bfloat16).contiguous()

    mpp = wl.max_pages_per_seq
    num_pages = B * mpp
    k_pool = torch.randn(num_pages, Hk, P, D, generator=g, device=dev, dtype=f32)
    v_pool = torch.randn(num_pages, Hk, P, D, generator=g, device=dev, dtype=f32)
    perm = torch.randperm(num_pages, generator=g, device=dev)
    page_table = perm.reshape(B, mpp).to(torch.int32)

    lens = list(wl.lens) if wl.lens is not None else [wl.L] * B
    heavy_all = []
    for b in range(B):
        L = lens[b]
        npg = (L + P - 1) // P
        if npg == 0:
            heavy_all.append([[] for _ in range(Hk)])
            continue
        coef = torch.zeros(Hk, npg * P, device=dev, dtype=f32)
        heavy_b = []
        for kvh in range(Hk):
            Bs = wl.block_sizes[kvh]
            j0, j1 = candidate_range(L, wl.S, wl.W, Bs)
            ncand = j1 - j0
            if wl.heavy_count is not None:
                nh = min(wl.heavy_count, ncand)
            else:
                nh = min(ncand, max(1, int(round(wl.heavy_frac * ncand))))
            picks = (torch.randperm(ncand, generator=g, device=dev)[:nh] + j0).tolist() if ncand else []
            picks = sorted(picks)
            heavy_b.append(picks)
            for j in picks:
                coef[kvh, j * Bs:(j + 1) * Bs] += wl.c_heavy
            if L > 0:
                coef[kvh, 0] += wl.c_sink
            if wl.recency > 0:
                r0 = max(0, L - wl.recency)
                n = L - r0
                coef[kvh, r0:L] += torch.linspace(0.0, 1.0, n, device=dev, dtype=f32)
        heavy_all.append(heavy_b)
        coef[:, L:] = 0.0
        rows = page_table[b, :npg].long()
        blk = k_pool[rows]                                          # [npg, Hk, P, D]
        add = coef.reshape(Hk, npg, P).permute(1, 0, 2).unsqueeze(-1) * g_hat[b].reshape(1, Hk, 1, D)
        k_pool[rows] = blk + add

    if wl.sink_heads > 0:
        q = q.reshape(B, Hq, D).clone()
        for b in range(B):
            picks = torch.randperm(Hq, generator=g, device=dev)[:wl.sink_heads].tolist()
            if lens[b] <= 0:
                continue
            row0 = int(page_table[b, 0])
            for h in picks:
                k0 = k_pool[row0, h // G, 0]
                q[b, h] += wl.c_qsink * k0 / k0.norm()
        q_bf = q.to(torch.bfloat16).contiguous()

    seq_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
    return DecodeCase(wl=wl, q=q_bf, k_pool=k_pool.to(torch.bfloat16),
                      v_pool=v_pool.to(torch.bfloat16), page_table=page_table,
                      seq_lens=seq_lens, g_hat=g_hat, heavy=heavy_all)


# --------------------------------------------------------------------------
# score-table workloads (table-driven selection over consecutive steps)
# --------------------------------------------------------------------------

@dataclass
class TableWorkload:
    """Consecutive decode steps whose candidates come from the score tables.

    Planted structure (a reading of the "drifting planted heavy positions" of
    the workload): per (sequence, KV group) n_vert heavy absolute positions in
    the middle region, one replaced every `drift` steps, plus heavy offsets
    from the newest token; each step's query leans on the keys there."""

    name: str
    B: int
    Hq: int
    Hk: int
    L0: int                         # tokens at the first step (current token included)
    steps: int
    S: int = 4
    W: int = 1024
    kcap: int = 6554
    beta: float = 1.0
    n_vert: int = 8
    slash_offsets: tuple = (2000, 5000, 20000, 60000)
    drift: int = 8
    c_q: float = 1.5
    t0_heavy: float = 0.02          # initial table value at planted entries
    t0_noise: float = 1e-5          # scale of the initial table elsewhere
    D: int = HEAD_DIM
    P: int = PAGE_SIZE

    @property
    def G(self):
        return self.Hq // self.Hk

    @property
    def max_pages_per_seq(self):
        return (self.L0 + self.steps + self.P - 1) // self.P


def table_workload(name: str) -> TableWorkload:
    if name == "tables_128k":
        # Llama-3-8B shape, batch 4, 131072 tokens growing by one per step
        return TableWorkload(name, B=4, Hq=32, Hk=8, L0=131072, steps=64)
    if name == "tables_small":
        return TableWorkload(name, B=2, Hq=8, Hk=2, L0=8192, steps=16, W=256, kcap=512, n_vert=4,
                             slash_offsets=(300, 1000, 4000, 7000), drift=4)
    raise KeyError(name)


@dataclass
class TableCase:
    wl: TableWorkload
    k_pool: torch.Tensor        # bf16 [num_pages, Hk, P, D]
    v_pool: torch.Tensor
    page_table: torch.Tensor    # int32 [B, max_pages]
    q_steps: torch.Tensor       # bf16 [steps, B, Hq, D]
    vert0: torch.Tensor         # fp32 [B, Hq, max_pages * P]
    slash0: torch.Tensor
    heavy: list                 # [step][b][kvh] -> positions


def make_table_case(wl: TableWorkload, seed: int, device="cpu") -> TableCase:
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(seed)
    B, Hq, Hk, G, D, P = wl.B, wl.Hq, wl.Hk, wl.G, wl.D, wl.P
    mpp = wl.max_pages_per_seq
    num_pages = B * mpp
    k_pool = torch.randn(num_pages, Hk, P, D, generator=g, device=dev).to(torch.bfloat16)
    v_pool = torch.randn(num_pages, Hk, P, D, generator=g, device=dev).to(torch.bfloat16)
    page_table = torch.randperm(num_pages, generator=g, device=dev).reshape(B, mpp).to(torch.int32)
    N = mpp * P
    lo_m, hi_m = wl.S, wl.L0 - wl.W
    heavy0 = torch.randint(lo_m, hi_m, (B, Hk, wl.n_vert), generator=g, device=dev)
    repl = torch.randint(lo_m, hi_m, (wl.steps // max(1, wl.drift) + 1, B, Hk), generator=g, device=dev)
    z = torch.randn(wl.steps, B, Hq, D, generator=g, device=dev)
    noise_v = torch.rand(B, Hq, N, generator=g, device=dev) * wl.t0_noise
    noise_s = torch.rand(B, Hq, N, generator=g, device=dev) * wl.t0_noise

    def key(b, kvh, pos):   # fp32 key rows of logical positions pos [n]
        pg = page_table[b, pos // P].long()
        return k_pool[pg, kvh, pos % P].float()

    heavy_steps = []
    cur = heavy0.clone()
    q = torch.empty(wl.steps, B, Hq, D, device=dev)
    for t in range(wl.steps):
        if t > 0 and wl.drift > 0 and t % wl.drift == 0:
            cur[:, :, (t // wl.drift - 1) % wl.n_vert] = repl[t // wl.drift]
        heavy_steps.append(cur.clone())
        L = wl.L0 + t
        for b in range(B):
            for kvh in range(Hk):
                pos_v = cur[b, kvh]
                pos_s = torch.tensor([L - 1 - d for d in wl.slash_offsets if L - 1 - d >= 0], device=dev)
                kk = torch.cat([key(b, kvh, pos_v), key(b, kvh, pos_s)])
                khat = kk / kk.norm(dim=-1, keepdim=True) * math.sqrt(D)
                lean = wl.c_q * khat.sum(dim=0)
                q[t, b, kvh * G:(kvh + 1) * G] = z[t, b, kvh * G:(kvh + 1) * G] + lean
    vert0 = noise_v.clone()
    slash0 = noise_s.clone()
    vert0[:, :, wl.L0:] = 0.0
    slash0[:, :, wl.L0:] = 0.0
    for b in range(B):
        for h in range(Hq):
            vert0[b, h, heavy0[b, h // G]] += wl.t0_heavy
            for d in wl.slash_offsets:
                if d < wl.L0:
                    slash0[b, h, d] += wl.t0_heavy
    return TableCase(wl=wl, k_pool=k_pool, v_pool=v_pool, page_table=page_table,
                     q_steps=q.to(torch.bfloat16), vert0=vert0.contiguous(), slash0=slash0.contiguous(),
                     heavy=[h.tolist() for h in heavy_steps])
