"""Shared test helpers: run the CUDA path through the binding and the oracle
on the same seeded inputs.  The oracle side only ever sees generator output."""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth

ATOL = 2e-3       # max-abs bound on O and lse
RTOL = 1e-2       # max-rel bound where |ref| >= 0.2
MODES = {"minmax": sa.SUMMARY_MINMAX, "mean": sa.SUMMARY_MEAN}


def assert_close(got: np.ndarray, ref: np.ndarray, what: str):
    """max-abs 2e-3 everywhere, and max-rel 1e-2 where |ref| >= 0.2; -inf must match."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    g, r = got[~inf_ref], ref[~inf_ref]
    if g.size == 0:
        return
    err = np.abs(g - r)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    i = int(np.argmax(err))
    assert err.max() <= ATOL, f"{what}: max abs err {err.max():.3e} at {i} (got {g[i]}, ref {r[i]})"
    big = np.abs(r) >= 0.2
    if big.any():
        rel = err[big] / np.abs(r[big])
        assert rel.max() <= RTOL, f"{what}: max rel err {rel.max():.3e}"


@dataclass
class NpCase:
    q: np.ndarray          # [B, Hq, D] float32 (bf16 values)
    k_pool: np.ndarray     # [num_pages, Hk, P, D] float32
    v_pool: np.ndarray
    page_table: np.ndarray  # [B, mpp]
    seq_lens: np.ndarray    # [B]


def to_np_case(case: synth.DecodeCase) -> NpCase:
    return NpCase(q=orc.to_np(case.q), k_pool=orc.to_np(case.k_pool), v_pool=orc.to_np(case.v_pool),
                  page_table=orc.to_np(case.page_table), seq_lens=orc.to_np(case.seq_lens))


def make_problem(wl: synth.Workload, ks: Sequence[int], kcap: Optional[int] = None,
                 mode: str = "minmax", num_pages: Optional[int] = None,
                 selection: int = sa.SELECT_PER_HEAD) -> sa.Problem:
    kc = max(1, max(ks)) if kcap is None else kcap
    npg = wl.B * wl.max_pages_per_seq if num_pages is None else num_pages
    return sa.Problem(B=wl.B, Hq=wl.Hq, Hk=wl.Hk, max_pages_per_seq=wl.max_pages_per_seq,
                      num_pages=npg, sink=wl.S, window=wl.W, block_sizes=wl.block_sizes,
                      k_per_head=list(ks), kcap=kc, mode=MODES[mode], selection=selection)


def to_dev(case: synth.DecodeCase, device="cuda"):
    return {n: getattr(case, n).to(device) for n in ("q", "k_pool", "v_pool", "page_table", "seq_lens")}


# ------------------------------------------------------------------ oracle side

def oracle_kv(nc: NpCase, b: int, kvh: int):
    L = int(nc.seq_lens[b])
    return (orc.gather_sequence(nc.k_pool, nc.page_table[b], kvh, L),
            orc.gather_sequence(nc.v_pool, nc.page_table[b], kvh, L))


def oracle_summaries(nc: NpCase, wl: synth.Workload, b: int, kvh: int, mode: str, j_begin=0, j_end=None):
    kseq, _ = oracle_kv(nc, b, kvh)
    return orc.summarize_sequence(kseq, wl.block_sizes[kvh], mode, j_begin, j_end)


def oracle_select(nc: NpCase, wl: synth.Workload, ks: Sequence[int], mode: str,
                  units: Optional[List[Tuple[int, int]]] = None):
    """{(b, h): (selected ascending, candidate ids, scores or None)}."""
    res = {}
    units = units if units is not None else [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    for b, kvh in units:
        kseq, _ = oracle_kv(nc, b, kvh)
        L = int(nc.seq_lens[b])
        Bs = wl.block_sizes[kvh]
        j0, j1 = orc.candidate_blocks(L, wl.S, wl.W, Bs)
        ids = np.arange(j0, j1, dtype=np.int64)
        summ = orc.summarize_sequence(kseq, Bs, mode, j0, j1) if j1 > j0 else None
        for g in range(wl.G):
            h = kvh * wl.G + g
            if j1 <= j0:
                res[(b, h)] = (np.zeros(0, np.int64), ids, np.zeros(0, np.float32))
                continue
            sc = orc.score_blocks(nc.q[b, h], summ, mode)
            res[(b, h)] = (orc.topk_blocks(sc, ids, ks[h]), ids, sc)
    return res


def oracle_select_group(nc: NpCase, wl: synth.Workload, ks: Sequence[int], mode: str,
                        units: Optional[List[Tuple[int, int]]] = None):
    """Group-shared selection: {(b, h): (selected ascending, candidate ids,
    group scores or None)}, the same entry for every head of a group."""
    res = {}
    units = units if units is not None else [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    for b, kvh in units:
        kseq, _ = oracle_kv(nc, b, kvh)
        L = int(nc.seq_lens[b])
        Bs = wl.block_sizes[kvh]
        q_group = [nc.q[b, kvh * wl.G + g] for g in range(wl.G)]
        r = orc.select_group(q_group, kseq, L, wl.S, wl.W, Bs, ks[kvh * wl.G], mode)
        for g in range(wl.G):
            res[(b, kvh * wl.G + g)] = r
    return res


def oracle_decode(nc: NpCase, wl: synth.Workload, sel: Dict[Tuple[int, int], np.ndarray], gran: int,
                  scale: float, units: Optional[List[Tuple[int, int]]] = None):
    """{(b, h): (O [D], lse)} for the given selections (block ids or token positions)."""
    out = {}
    units = units if units is not None else [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    for b, kvh in units:
        kseq, vseq = oracle_kv(nc, b, kvh)
        L = int(nc.seq_lens[b])
        for g in range(wl.G):
            h = kvh * wl.G + g
            s = sel.get((b, h), np.zeros(0, np.int64))
            if gran == sa.SEL_BLOCK:
                r = orc.decode_head(nc.q[b, h], kseq, vseq, L, wl.S, wl.W, wl.block_sizes[kvh], s, scale)
                out[(b, h)] = (r["O"], r["lse"])
            else:
                s_end, w_beg = orc.partition(L, wl.S, wl.W)
                J = np.array(sorted(set(int(t) for t in s if s_end <= t < w_beg)), dtype=np.int64)
                I = orc.dense_tokens(L, wl.S, wl.W)
                O_I, l_I = orc.attend(nc.q[b, h], kseq, vseq, I, scale)
                O_J, l_J = orc.attend(nc.q[b, h], kseq, vseq, J, scale)
                O, lse = orc.lse_merge(O_I, l_I, O_J, l_J)
                out[(b, h)] = (O, float(lse))
    return out


def oracle_bypass(nc: NpCase, wl: synth.Workload, scale: float, units: Optional[List[Tuple[int, int]]] = None):
    """{(b, h): (rho, lse_est, mean value row)} of the head-sparsity estimate."""
    res = {}
    units = units if units is not None else [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    for b, kvh in units:
        kseq, vseq = oracle_kv(nc, b, kvh)
        L = int(nc.seq_lens[b])
        vbar = orc.bypass_output(vseq, L)
        for g in range(wl.G):
            h = kvh * wl.G + g
            rho, lse = orc.head_sparsity(nc.q[b, h], kseq, L, scale)
            res[(b, h)] = (rho, lse, vbar)
    return res


def oracle_kv_stats(nc: NpCase, b: int, kvh: int):
    """fp64 sums of k, k*k and v over the sequence, and of |k|, k*k, |v| (the error scale)."""
    kseq, vseq = oracle_kv(nc, b, kvh)
    k, v = kseq.astype(np.float64), vseq.astype(np.float64)
    sums = np.stack([k.sum(0), (k * k).sum(0), v.sum(0)])
    mags = np.stack([np.abs(k).sum(0), (k * k).sum(0), np.abs(v).sum(0)])
    return sums, mags


# ------------------------------------------------------------------ GPU side

def gpu_summaries(prob: sa.Problem, dev, ws):
    summ = torch.zeros(prob.summary_shape(), dtype=torch.bfloat16, device="cuda")
    sa.block_summarize(prob, dev["k_pool"], dev["page_table"], dev["seq_lens"], summ, ws)
    return summ


def gpu_select(prob: sa.Problem, dev, summ, ws, with_scores=True):
    sel_idx = torch.full((prob.B, prob.Hq, prob.kcap), -7, dtype=torch.int32, device="cuda")
    sel_cnt = torch.full((prob.B, prob.Hq), -7, dtype=torch.int32, device="cuda")
    scores = torch.full((prob.B, prob.Hq, prob.block_slots()), float("nan"), device="cuda") if with_scores else None
    sa.select_topk(prob, dev["q"], summ, dev["seq_lens"], sel_idx, sel_cnt, ws, scores)
    return sel_idx, sel_cnt, scores


def sel_to_tensor(prob: sa.Problem, sel: Dict[Tuple[int, int], np.ndarray]):
    idx = torch.full((prob.B, prob.Hq, prob.kcap), -1, dtype=torch.int32)
    cnt = torch.zeros((prob.B, prob.Hq), dtype=torch.int32)
    for (b, h), s in sel.items():
        s = np.asarray(s, np.int64)
        assert len(s) <= prob.kcap
        idx[b, h, :len(s)] = torch.from_numpy(s.astype(np.int32))
        cnt[b, h] = len(s)
    return idx.cuda(), cnt.cuda()


def gpu_decode(prob: sa.Problem, dev, sel_idx, sel_cnt, ws, gran=sa.SEL_BLOCK, logits=None):
    out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
    lse = torch.full((prob.B, prob.Hq), float("nan"), device="cuda")
    sa.sparse_decode(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"],
                     sel_idx, sel_cnt, out, lse, ws, granularity=gran, logits=logits)
    return out, lse
