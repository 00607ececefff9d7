"""Timing of the oracle on host cores (test infrastructure: used only by the
benchmark's CPU-baseline leg and its reference arm).

The oracle runs as it stands -- the same calls the parity tests make -- over
whole units of one decode step:
  - "decode": one (sequence, KV head) of block selection plus attention:
    per head the canonical-fp32 block scores and top-k, then the fp64
    attention over the dense set and the selected blocks with the exact
    log-sum-exp merge;
  - "table": one query head of a score-table step: the fp64 table update
    from the previous step's merged weights, the threshold and expansion of
    the candidates, and the fp64 attention over the dense set plus them.
Units run one after another in this process (one core) or spread over a
spawn-started process pool (all cores).  The KV pools reach the workers
as raw bf16 bits in memory-mapped files; nothing here imports the CUDA
binding.
"""
from __future__ import annotations

import math
import multiprocessing as mp
import os
import shutil
import tempfile
import time
from typing import Dict, List, Optional, Sequence

import numpy as np

from oracle import sparse_attention_oracle as orc

# ------------------------------------------------------------------ shared pools

_attached: Dict[str, tuple] = {}


class SharedPools:
    """bf16 K / V pools (as uint16 bits) in memory-mapped temporary files,
    shared with the workers through the page cache (no /dev/shm needed)."""

    def __init__(self, k_bits: np.ndarray, v_bits: np.ndarray):
        self.shape = tuple(k_bits.shape)
        self.dir = tempfile.mkdtemp(prefix="sa_oracle_")
        self.paths = []
        for nm, a in (("k", k_bits), ("v", v_bits)):
            path = os.path.join(self.dir, nm + ".u16")
            m = np.memmap(path, dtype=np.uint16, mode="w+", shape=self.shape)
            m[...] = a
            m.flush()
            del m
            self.paths.append(path)
        self.local = [np.memmap(pth, dtype=np.uint16, mode="r", shape=self.shape) for pth in self.paths]

    def spec(self):
        return {"paths": list(self.paths), "shape": self.shape}

    def close(self):
        self.local = []
        shutil.rmtree(self.dir, ignore_errors=True)


def _pools(spec, local=None):
    if local is not None:
        return local
    key = spec["paths"][0]
    if key not in _attached:
        _attached.clear()
        _attached[key] = [np.memmap(pth, dtype=np.uint16, mode="r", shape=tuple(spec["shape"]))
                          for pth in spec["paths"]]
    return _attached[key]


def _seq_f32(pool_bits: np.ndarray, page_row: np.ndarray, kvh: int, L: int) -> np.ndarray:
    """fp32 rows [L, D] of one sequence of one KV head (bf16 bits widened)."""
    bits = orc.gather_sequence(pool_bits, page_row, kvh, L)
    return (bits.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ units

def decode_unit(job, local=None) -> float:
    """One (sequence, KV head) of a block-selection step; returns seconds."""
    kb, vb = _pools(job["pools"], local)
    t0 = time.perf_counter()
    L, S, W, Bs = job["L"], job["S"], job["W"], job["Bs"]
    kseq = _seq_f32(kb, job["page_row"], job["kvh"], L)
    vseq = _seq_f32(vb, job["page_row"], job["kvh"], L)
    j0, j1 = orc.candidate_blocks(L, S, W, Bs)
    ids = np.arange(j0, j1, dtype=np.int64)
    summ = orc.summarize_sequence(kseq, Bs, job["mode"], j0, j1) if j1 > j0 else None
    for q, k in zip(job["q"], job["k"]):
        sel = np.zeros(0, np.int64)
        if j1 > j0:
            sel = orc.topk_blocks(orc.score_blocks(q, summ, job["mode"]), ids, k)
        orc.decode_head(q, kseq, vseq, L, S, W, Bs, sel, job["scale"])
    return time.perf_counter() - t0


def table_unit(job, local=None) -> float:
    """One query head of a score-table step (update, candidates, attention)."""
    kb, vb = _pools(job["pools"], local)
    t0 = time.perf_counter()
    L0, S, W = job["L0"], job["S"], job["W"]
    L = L0 + 1
    kseq = _seq_f32(kb, job["page_row"], job["kvh"], L)
    vseq = _seq_f32(vb, job["page_row"], job["kvh"], L)
    c0, _ = orc.table_candidates(job["vert"], job["slash"], L0, S, W, job["beta"], job["kcap"])
    pos, w = orc.merged_weights(job["q_prev"], kseq, L0, S, W, c0, job["scale"])
    v1, s1 = orc.table_update(job["vert"], job["slash"], L0, pos, w)
    c1, _ = orc.table_candidates(v1.astype(np.float32), s1.astype(np.float32), L, S, W, job["beta"], job["kcap"])
    I = orc.dense_tokens(L, S, W)
    O_I, l_I = orc.attend(job["q"], kseq, vseq, I, job["scale"])
    O_J, l_J = orc.attend(job["q"], kseq, vseq, c1, job["scale"])
    orc.lse_merge(O_I, l_I, O_J, l_J)
    return time.perf_counter() - t0


def _run_job(job):
    return (decode_unit if job["kind"] == "decode" else table_unit)(job)


# ------------------------------------------------------------------ jobs of a case

def decode_jobs(pools_spec, q: np.ndarray, page_table: np.ndarray, seq_lens: Sequence[int], block_sizes, ks,
                S: int, W: int, mode: str, scale: float, units=None) -> List[dict]:
    """Jobs of a block-selection step; q fp32 [B, Hq, D]."""
    B, Hq = q.shape[0], q.shape[1]
    Hk = len(block_sizes)
    G = Hq // Hk
    units = units if units is not None else [(b, kvh) for b in range(B) for kvh in range(Hk)]
    return [dict(kind="decode", pools=pools_spec, page_row=page_table[b], kvh=kvh, L=int(seq_lens[b]), S=S, W=W,
                 Bs=int(block_sizes[kvh]), mode=mode, scale=scale,
                 q=[q[b, kvh * G + g] for g in range(G)], k=[int(ks[kvh * G + g]) for g in range(G)])
            for (b, kvh) in units]


def table_jobs(pools_spec, q_prev, q_cur, page_table, vert, slash, L0: int, S: int, W: int, beta: float,
               kcap: int, G: int, scale: float, heads) -> List[dict]:
    """Jobs of one score-table step for the given (sequence, query head)s."""
    return [dict(kind="table", pools=pools_spec, page_row=page_table[b], kvh=h // G, L0=L0, S=S, W=W, beta=beta,
                 kcap=kcap, scale=scale, q_prev=q_prev[b, h], q=q_cur[b, h], vert=vert[b, h], slash=slash[b, h])
            for (b, h) in heads]


# ------------------------------------------------------------------ timing

def cores_available() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OraclePool:
    """A spawn-started pool of `cores` workers (safe after CUDA has been
    initialised in the parent: nothing is forked)."""

    _ONE_THREAD = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")

    def __init__(self, cores: Optional[int] = None):
        self.cores = cores or cores_available()
        # one BLAS thread per worker process: the pool is the parallelism
        saved = {k: os.environ.get(k) for k in self._ONE_THREAD}
        for k in self._ONE_THREAD:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(self.cores)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.pool.map(math.sqrt, range(self.cores))   # start every worker before timing

    def close(self):
        self.pool.close()
        self.pool.join()


def time_serial(jobs: List[dict], local_pools, budget_s: float):
    """Run jobs in order on this core until the budget is spent; returns
    (seconds, jobs done)."""
    t0 = time.perf_counter()
    n = 0
    for j in jobs:
        (decode_unit if j["kind"] == "decode" else table_unit)(j, local_pools)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    return time.perf_counter() - t0, n


def time_parallel(pool: OraclePool, jobs: List[dict]):
    """Run all jobs over the pool; returns wall seconds."""
    t0 = time.perf_counter()
    pool.pool.map(_run_job, jobs, chunksize=1)
    return time.perf_counter() - t0
