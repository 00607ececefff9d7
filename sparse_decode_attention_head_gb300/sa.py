"""Thin ctypes binding of libsa (include/sa.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (device memory and streams come from
PyTorch); each call launches on torch's current stream.  There is no CPU
fallback: if libsa.so is missing or no GPU is present the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import List, Optional, Sequence

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libsa.so")
HEADER = os.path.join(ROOT, "include", "sa.h")

SA_OK = 0
SA_ERR_INVALID_ARG = 1
SA_ERR_UNSUPPORTED = 2
SA_ERR_CUDA = 3
SA_ERR_CAPACITY = 4
SA_ERR_BAD_PAGE = 5
SA_ERR_TIMEOUT = 6
SUMMARY_MINMAX = 0
SUMMARY_MEAN = 1
SEL_BLOCK = 0
SEL_TOKEN = 1
SELECT_PER_HEAD = 0
SELECT_GROUP = 1
BLOCKS_TAIL = -1
HEAD_DIM = 128
PAGE_SIZE = 16


class SAError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} (code {code})")
        self.code = code


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hk", ctypes.c_int32), ("D", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("sink", ctypes.c_int32), ("window", ctypes.c_int32), ("summary_mode", ctypes.c_int32),
        ("block_size_per_kvh", ctypes.POINTER(ctypes.c_int32)), ("k_per_qhead", ctypes.POINTER(ctypes.c_int32)),
        ("kcap", ctypes.c_int32), ("scale", ctypes.c_float), ("selection_mode", ctypes.c_int32),
    ]


_lib = None


def lib():
    """Load libsa.so (built in-tree by build_lib.build())."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with sparse_decode_attention_head_gb300.build_lib.build()")
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(_Problem)
        vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        sig = {
            "sa_block_slots": (i32, [P]),
            "sa_workspace_size": (sz, [P]),
            "sa_workspace_init": (ctypes.c_int, [vp, sz, vp]),
            "sa_get_status": (ctypes.c_int, [vp, vp, ctypes.POINTER(ctypes.c_int)]),
            "sa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "sa_block_summarize": (ctypes.c_int, [P, vp, vp, vp, i32, i32, vp, vp, vp]),
            "sa_score_blocks": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp]),
            "sa_select_topk": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_sparse_decode": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]),
            "sa_lse_merge": (ctypes.c_int, [i32, i32, vp, vp, vp, vp, vp, vp, vp]),
            "sa_sparse_decode_noalloc": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, vp]),
            "sa_decode_step": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_select_tokens": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_append_kv": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_decode_step_append": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_update_score_tables": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                      ctypes.c_float, ctypes.c_float, vp, vp, vp, vp]),
            "sa_kv_stats": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp]),
            "sa_head_sparsity": (ctypes.c_int, [P, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, vp, vp]),
            "sa_decode_step_bypass": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float,
                                                     vp, vp, vp, vp, vp, vp, vp, vp]),
            "sa_step_plan_create": (ctypes.c_int, [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                   ctypes.POINTER(vp)]),
            "sa_step_plan_launch": (ctypes.c_int, [vp, vp]),
            "sa_step_plan_destroy": (ctypes.c_int, [vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions() -> List[str]:
    """Names of the functions declared in include/sa.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(sa_[a-z_0-9]+)\s*\(", txt)))


def status_string(code: int) -> str:
    try:
        return lib().sa_status_string(int(code)).decode()
    except Exception:
        return "unknown"


def _check(rc: int, what: str):
    if rc != SA_OK:
        raise SAError(rc, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class Problem:
    """Shapes and selection settings of one attention layer (sa_problem)."""

    def __init__(self, B: int, Hq: int, Hk: int, max_pages_per_seq: int, num_pages: int, sink: int,
                 window: int, block_sizes: Sequence[int], k_per_head: Sequence[int], kcap: int,
                 mode: int = SUMMARY_MINMAX, scale: Optional[float] = None, D: int = HEAD_DIM,
                 page_size: int = PAGE_SIZE, selection: int = SELECT_PER_HEAD):
        self.B, self.Hq, self.Hk, self.D = B, Hq, Hk, D
        self.max_pages_per_seq, self.num_pages = max_pages_per_seq, num_pages
        self.sink, self.window, self.mode, self.kcap = sink, window, mode, kcap
        self.page_size = page_size
        self.scale = 1.0 / math.sqrt(D) if scale is None else scale
        self.block_sizes = list(block_sizes)
        self.k_per_head = list(k_per_head)
        self._bs = (ctypes.c_int32 * max(1, len(self.block_sizes)))(*self.block_sizes)
        self._k = (ctypes.c_int32 * max(1, len(self.k_per_head)))(*self.k_per_head)
        self._summary_shape = None
        self._c = _Problem(B, Hq, Hk, D, page_size, max_pages_per_seq, num_pages, sink, window, mode,
                           ctypes.cast(self._bs, ctypes.POINTER(ctypes.c_int32)),
                           ctypes.cast(self._k, ctypes.POINTER(ctypes.c_int32)), kcap, self.scale, selection)
        self.selection = selection

    @property
    def G(self):
        return self.Hq // self.Hk

    @property
    def ref(self):
        return ctypes.byref(self._c)

    def block_slots(self) -> int:
        return int(lib().sa_block_slots(self.ref))

    def workspace_size(self) -> int:
        return int(lib().sa_workspace_size(self.ref))

    def summary_shape(self):
        if self._summary_shape is None:
            s = self.block_slots()
            if self.mode == SUMMARY_MINMAX:
                self._summary_shape = (self.B, self.Hk, s, 2, self.D)
            else:
                self._summary_shape = (self.B, self.Hk, s, self.D)
        return self._summary_shape


class Workspace:
    """Device scratch for one problem (sa_workspace_size bytes), zeroed once."""

    def __init__(self, prob: Problem, device="cuda"):
        n = prob.workspace_size()
        if n == 0:
            raise SAError(SA_ERR_INVALID_ARG, "sa_workspace_size")
        self.buf = torch.empty(n, dtype=torch.uint8, device=device)
        _check(lib().sa_workspace_init(_ptr(self.buf), n, _stream()), "sa_workspace_init")

    def status(self) -> int:
        v = ctypes.c_int(0)
        _check(lib().sa_get_status(_ptr(self.buf), _stream(), ctypes.byref(v)), "sa_get_status")
        return v.value


def block_summarize(prob: Problem, k_pool, page_table, seq_lens, summaries, ws: Workspace,
                    block_begin: int = 0, block_end: int = -1):
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(summaries, torch.bfloat16, "summaries", prob.summary_shape())
    _check(lib().sa_block_summarize(prob.ref, _ptr(k_pool), _ptr(page_table), _ptr(seq_lens), block_begin,
                                    block_end, _ptr(summaries), _ptr(ws.buf), _stream()), "sa_block_summarize")


def score_blocks(prob: Problem, q, summaries, seq_lens, scores, ws: Workspace):
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(summaries, torch.bfloat16, "summaries", prob.summary_shape())
    _need(scores, torch.float32, "scores", (prob.B, prob.Hq, prob.block_slots()))
    _check(lib().sa_score_blocks(prob.ref, _ptr(q), _ptr(summaries), _ptr(seq_lens), _ptr(scores),
                                 _ptr(ws.buf), _stream()), "sa_score_blocks")


def select_topk(prob: Problem, q, summaries, seq_lens, sel_idx, sel_cnt, ws: Workspace, scores=None):
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(summaries, torch.bfloat16, "summaries", prob.summary_shape())
    _need(sel_idx, torch.int32, "sel_idx", (prob.B, prob.Hq, prob.kcap))
    _need(sel_cnt, torch.int32, "sel_cnt", (prob.B, prob.Hq))
    if scores is not None:
        _need(scores, torch.float32, "scores", (prob.B, prob.Hq, prob.block_slots()))
    _check(lib().sa_select_topk(prob.ref, _ptr(q), _ptr(summaries), _ptr(seq_lens), _ptr(sel_idx),
                                _ptr(sel_cnt), _ptr(scores), _ptr(ws.buf), _stream()), "sa_select_topk")


def sparse_decode(prob: Problem, q, k_pool, v_pool, page_table, seq_lens, sel_idx, sel_cnt, out, lse,
                  ws: Workspace, granularity: int = SEL_BLOCK, logits=None, bypass=None):
    """bypass: optional [B][Hq] int32 flags of sa_head_sparsity; flagged heads
    are left out and their out / lse rows are not written."""
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool", tuple(k_pool.shape))
    if k_pool.shape[0] != prob.num_pages or k_pool.shape[1:] != (prob.Hk, prob.page_size, prob.D):
        raise ValueError("pools must be [num_pages][Hk][page_size][D]")
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(sel_idx, torch.int32, "sel_idx", (prob.B, prob.Hq, prob.kcap))
    _need(sel_cnt, torch.int32, "sel_cnt", (prob.B, prob.Hq))
    _need(out, torch.float32, "out", (prob.B, prob.Hq, prob.D))
    _need(lse, torch.float32, "lse", (prob.B, prob.Hq))
    if logits is not None:
        _need(logits, torch.float32, "logits", (prob.B, prob.Hq, prob.max_pages_per_seq * prob.page_size))
    if bypass is not None:
        _need(bypass, torch.int32, "bypass", (prob.B, prob.Hq))
    _check(lib().sa_sparse_decode(prob.ref, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                  _ptr(seq_lens), _ptr(sel_idx), _ptr(sel_cnt), granularity, _ptr(out),
                                  _ptr(lse), _ptr(logits), _ptr(bypass), _ptr(ws.buf), _stream()),
           "sa_sparse_decode")


def lse_merge(o_a, lse_a, o_b, lse_b, o, lse):
    n, D = o_a.shape
    for t, nm in ((o_a, "o_a"), (o_b, "o_b"), (o, "o")):
        _need(t, torch.float32, nm, (n, D))
    for t, nm in ((lse_a, "lse_a"), (lse_b, "lse_b"), (lse, "lse")):
        _need(t, torch.float32, nm, (n,))
    _check(lib().sa_lse_merge(n, D, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o), _ptr(lse),
                              _stream()), "sa_lse_merge")


def update_score_tables(prob: Problem, vert_in, slash_in, vert_out, slash_out, seq_lens, cand_idx, cand_cnt,
                        ws: Workspace, decay: float = 0.95, beta: float = 1.0, prev=None, prev_bypass=None):
    """prev: None (first step: tables copied) or a dict with prev_seq_lens,
    prev_sel_idx, prev_sel_cnt, prev_logits, prev_lse of the previous step.
    prev_bypass: optional [B][Hq] int32 flags of the previous step's
    sa_head_sparsity; the tables of flagged heads are copied unchanged."""
    N = prob.max_pages_per_seq * prob.page_size
    for t, nm in ((vert_in, "vert_in"), (slash_in, "slash_in"), (vert_out, "vert_out"), (slash_out, "slash_out")):
        _need(t, torch.float32, nm, (prob.B, prob.Hq, N))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(cand_idx, torch.int32, "cand_idx", (prob.B, prob.Hq, prob.kcap))
    _need(cand_cnt, torch.int32, "cand_cnt", (prob.B, prob.Hq))
    pv = prev or {}
    if prev is not None:
        _need(pv["prev_seq_lens"], torch.int32, "prev_seq_lens", (prob.B,))
        _need(pv["prev_sel_idx"], torch.int32, "prev_sel_idx", (prob.B, prob.Hq, prob.kcap))
        _need(pv["prev_sel_cnt"], torch.int32, "prev_sel_cnt", (prob.B, prob.Hq))
        _need(pv["prev_logits"], torch.float32, "prev_logits", (prob.B, prob.Hq, N))
        _need(pv["prev_lse"], torch.float32, "prev_lse", (prob.B, prob.Hq))
    if prev_bypass is not None:
        _need(prev_bypass, torch.int32, "prev_bypass", (prob.B, prob.Hq))
    _check(lib().sa_update_score_tables(
        prob.ref, _ptr(vert_in), _ptr(slash_in), _ptr(vert_out), _ptr(slash_out), _ptr(pv.get("prev_seq_lens")),
        _ptr(pv.get("prev_sel_idx")), _ptr(pv.get("prev_sel_cnt")), _ptr(pv.get("prev_logits")),
        _ptr(pv.get("prev_lse")), _ptr(prev_bypass), _ptr(seq_lens), decay, beta, _ptr(cand_idx), _ptr(cand_cnt), _ptr(ws.buf),
        _stream()), "sa_update_score_tables")


def select_tokens(prob: Problem, q, k_pool, page_table, seq_lens, cand_idx, cand_cnt, sel_idx, sel_cnt,
                  ws: Workspace, scores=None):
    """Exact top-k inside the score-table candidates (sa_select_tokens): the
    k_per_head[h] best candidate tokens by the canonical fp32 q . k."""
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    for t, nm in ((cand_idx, "cand_idx"), (sel_idx, "sel_idx")):
        _need(t, torch.int32, nm, (prob.B, prob.Hq, prob.kcap))
    for t, nm in ((cand_cnt, "cand_cnt"), (sel_cnt, "sel_cnt")):
        _need(t, torch.int32, nm, (prob.B, prob.Hq))
    if scores is not None:
        _need(scores, torch.float32, "scores", (prob.B, prob.Hq, prob.kcap))
    _check(lib().sa_select_tokens(prob.ref, _ptr(q), _ptr(k_pool), _ptr(page_table), _ptr(seq_lens), _ptr(cand_idx),
                                  _ptr(cand_cnt), _ptr(sel_idx), _ptr(sel_cnt), _ptr(scores), _ptr(ws.buf),
                                  _stream()), "sa_select_tokens")


def _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse):
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool", tuple(k_pool.shape))
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(summaries, torch.bfloat16, "summaries", prob.summary_shape())
    _need(sel_idx, torch.int32, "sel_idx", (prob.B, prob.Hq, prob.kcap))
    _need(sel_cnt, torch.int32, "sel_cnt", (prob.B, prob.Hq))
    _need(out, torch.float32, "out", (prob.B, prob.Hq, prob.D))
    _need(lse, torch.float32, "lse", (prob.B, prob.Hq))


def decode_step(prob: Problem, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse,
                ws: Workspace):
    """Whole block-selection decode step: tail-block summary refresh, scores,
    top-k and the paged sparse decode (sa_decode_step)."""
    _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse)
    _check(lib().sa_decode_step(prob.ref, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens),
                                _ptr(summaries), _ptr(sel_idx), _ptr(sel_cnt), _ptr(out), _ptr(lse), _ptr(ws.buf),
                                _stream()), "sa_decode_step")


def append_kv(prob: Problem, k_new, v_new, k_pool, v_pool, page_table, seq_lens, ws: Workspace):
    """The new token's K and V rows into the pools at position seq_lens[b] - 1 (sa_append_kv)."""
    for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, nm, (prob.B, prob.Hk, prob.D))
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool", tuple(k_pool.shape))
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _check(lib().sa_append_kv(prob.ref, _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                              _ptr(seq_lens), _ptr(ws.buf), _stream()), "sa_append_kv")


def decode_step_append(prob: Problem, q, k_new, v_new, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx,
                       sel_cnt, out, lse, ws: Workspace):
    """The new token's K/V appended, then the whole decode step (sa_decode_step_append)."""
    _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse)
    for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.bfloat16, nm, (prob.B, prob.Hk, prob.D))
    _check(lib().sa_decode_step_append(prob.ref, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                       _ptr(page_table), _ptr(seq_lens), _ptr(summaries), _ptr(sel_idx),
                                       _ptr(sel_cnt), _ptr(out), _ptr(lse), _ptr(ws.buf), _stream()),
           "sa_decode_step_append")


BYPASS_EPS = 0.85   # LFPS's sparsity threshold epsilon


def kv_stats_shape(prob: Problem):
    return (prob.B, prob.Hk, 3, prob.D)


def kv_stats(prob: Problem, k_pool, v_pool, page_table, seq_lens, stats, ws: Workspace):
    """Per (b, KV head) fp32 sums of k, k*k and v over the cached tokens (sa_kv_stats)."""
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(v_pool, torch.bfloat16, "v_pool", tuple(k_pool.shape))
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(stats, torch.float32, "kv_stats", kv_stats_shape(prob))
    _check(lib().sa_kv_stats(prob.ref, _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens), _ptr(stats),
                             _ptr(ws.buf), _stream()), "sa_kv_stats")


def head_sparsity(prob: Problem, q, k_pool, page_table, seq_lens, stats, bypass, out, lse, ws: Workspace,
                  eps: float = BYPASS_EPS, rho=None):
    """LFPS's sink-share estimate per head and the mean-value bypass
    (sa_head_sparsity): bypass[b][h] = rho > eps; bypassed rows of out / lse
    receive the mean value row and the estimated log-normaliser."""
    _need(q, torch.bfloat16, "q", (prob.B, prob.Hq, prob.D))
    _need(k_pool, torch.bfloat16, "k_pool")
    _need(page_table, torch.int32, "page_table", (prob.B, prob.max_pages_per_seq))
    _need(seq_lens, torch.int32, "seq_lens", (prob.B,))
    _need(stats, torch.float32, "kv_stats", kv_stats_shape(prob))
    _need(bypass, torch.int32, "bypass", (prob.B, prob.Hq))
    _need(out, torch.float32, "out", (prob.B, prob.Hq, prob.D))
    _need(lse, torch.float32, "lse", (prob.B, prob.Hq))
    if rho is not None:
        _need(rho, torch.float32, "rho", (prob.B, prob.Hq))
    _check(lib().sa_head_sparsity(prob.ref, _ptr(q), _ptr(k_pool), _ptr(page_table), _ptr(seq_lens), _ptr(stats),
                                  float(eps), _ptr(rho), _ptr(bypass), _ptr(out), _ptr(lse), _ptr(ws.buf),
                                  _stream()), "sa_head_sparsity")


def decode_step_bypass(prob: Problem, q, k_pool, v_pool, page_table, seq_lens, summaries, stats, sel_idx, sel_cnt,
                       out, lse, bypass, ws: Workspace, eps: float = BYPASS_EPS, rho=None, k_new=None, v_new=None):
    """The decode step with LFPS's head-sparsity bypass (sa_decode_step_bypass);
    with k_new / v_new the new token is appended first and added to stats."""
    _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse)
    _need(stats, torch.float32, "kv_stats", kv_stats_shape(prob))
    _need(bypass, torch.int32, "bypass", (prob.B, prob.Hq))
    if rho is not None:
        _need(rho, torch.float32, "rho", (prob.B, prob.Hq))
    if (k_new is None) != (v_new is None):
        raise ValueError("k_new and v_new go together")
    if k_new is not None:
        for t, nm in ((k_new, "k_new"), (v_new, "v_new")):
            _need(t, torch.bfloat16, nm, (prob.B, prob.Hk, prob.D))
    _check(lib().sa_decode_step_bypass(prob.ref, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_pool), _ptr(v_pool),
                                       _ptr(page_table), _ptr(seq_lens), _ptr(summaries), _ptr(stats), float(eps),
                                       _ptr(sel_idx), _ptr(sel_cnt), _ptr(out), _ptr(lse), _ptr(rho), _ptr(bypass),
                                       _ptr(ws.buf), _stream()), "sa_decode_step_bypass")


class DecodeStepCall:
    """sa_decode_step bound to fixed tensors: the arguments are checked and
    marshalled once, each call passes only the current stream.  The tensors'
    contents may change between calls (a serving loop that reuses its
    buffers); the object keeps them alive."""

    def __init__(self, prob: Problem, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out,
                 lse, ws: Workspace):
        _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse)
        self._keep = (prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse, ws)
        self._fn = lib().sa_decode_step
        self._args = (prob.ref, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table), _ptr(seq_lens),
                      _ptr(summaries), _ptr(sel_idx), _ptr(sel_cnt), _ptr(out), _ptr(lse), _ptr(ws.buf))

    def __call__(self):
        rc = self._fn(*self._args, _stream())
        if rc != SA_OK:
            raise SAError(rc, "sa_decode_step")


class StepPlan:
    """sa_decode_step on fixed tensors, prepared once as a CUDA graph inside
    the library (sa_step_plan_create); each call replays it on the current
    stream with one graph launch (sa_step_plan_launch).  The tensors'
    contents may change between calls; the object keeps them alive and frees
    the plan when it is collected or closed."""

    def __init__(self, prob: Problem, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out,
                 lse, ws: Workspace):
        _check_step_args(prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse)
        self._keep = (prob, q, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt, out, lse, ws)
        self._lib = lib()
        h = ctypes.c_void_p()
        _check(self._lib.sa_step_plan_create(prob.ref, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(page_table),
                                             _ptr(seq_lens), _ptr(summaries), _ptr(sel_idx), _ptr(sel_cnt),
                                             _ptr(out), _ptr(lse), _ptr(ws.buf), ctypes.byref(h)),
               "sa_step_plan_create")
        self._h = h
        self._launch = self._lib.sa_step_plan_launch

    def __call__(self):
        rc = self._launch(self._h, _stream())
        if rc != SA_OK:
            raise SAError(rc, "sa_step_plan_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.sa_step_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
