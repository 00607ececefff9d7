"""Parity of the CUDA path (through the C-ABI) against the fp64 oracle.

Index sets and block scores must match bit for bit; O and lse within max-abs
2e-3 (and max-rel 1e-2 where |ref| >= 0.2), given the same index set."""
import math

import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sa.lib()


def _check_selection(prob, wl, nc, sel_idx, sel_cnt, scores, ref, units=None):
    si, sc_ = sel_idx.cpu().numpy(), sel_cnt.cpu().numpy()
    sco = scores.cpu().numpy() if scores is not None else None
    for (b, h), (sel, ids, osc) in ref.items():
        n = int(sc_[b, h])
        assert n == len(sel), f"(b={b}, h={h}) count {n} vs {len(sel)}"
        assert np.array_equal(si[b, h, :n], sel), f"(b={b}, h={h}) index set differs"
        if sco is not None and osc is not None and len(ids):
            got = sco[b, h, ids]
            assert np.array_equal(got.view(np.uint32), osc.astype(np.float32).view(np.uint32)), \
                f"(b={b}, h={h}) scores differ (max diff {np.max(np.abs(got - osc))})"


def _check_decode(out, lse, ref):
    o, l = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), (O, lz) in ref.items():
        H.assert_close(o[b, h], O, f"O(b={b},h={h})")
        H.assert_close(np.array([l[b, h]]), np.array([lz]), f"lse(b={b},h={h})")


def _full_pipeline(wl, seed, mode, units=None, check_summaries=True, ks=None):
    case = synth.make_decode_case(wl, seed)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl) if ks is None else ks
    prob = H.make_problem(wl, ks, mode=mode)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    if check_summaries:
        sg = summ.float().cpu().numpy()
        for b, kvh in (units or [(b, k) for b in range(wl.B) for k in range(wl.Hk)]):
            L = int(nc.seq_lens[b])
            nb = -(-L // wl.block_sizes[kvh])
            ref = H.oracle_summaries(nc, wl, b, kvh, mode)
            assert np.array_equal(sg[b, kvh, :nb], ref), f"summaries differ at b={b} kvh={kvh}"
    sel_idx, sel_cnt, scores = H.gpu_select(prob, dev, summ, ws)
    ref_sel = H.oracle_select(nc, wl, ks, mode, units)
    _check_selection(prob, wl, nc, sel_idx, sel_cnt, scores, ref_sel)
    out, lse = H.gpu_decode(prob, dev, sel_idx, sel_cnt, ws)
    ref_dec = H.oracle_decode(nc, wl, {k: v[0] for k, v in ref_sel.items()}, sa.SEL_BLOCK, prob.scale, units)
    _check_decode(out, lse, ref_dec)
    assert ws.status() == sa.SA_OK
    return prob, dev, ws, nc, ref_sel


@pytest.mark.parametrize("mode", ["minmax", "mean"])
def test_tiny_4k_end_to_end(mode):
    _full_pipeline(synth.workload("tiny_4k"), 0, mode)


@pytest.mark.parametrize("mode", ["minmax", "mean"])
def test_llama_32k_full_size(mode):
    # every (sequence, head) of the Llama-shaped 32K layer, at full size
    _full_pipeline(synth.workload("llama_32k"), 1, mode)


def test_qwen_64k_head_specific_sampled():
    wl = synth.workload("qwen_64k")
    units = [(0, 0), (5, 1), (11, 2), (15, 3)]
    _full_pipeline(wl, 2, "minmax", units=units)


def _small(name="small", **kw):
    base = dict(B=3, Hq=6, Hk=2, L=1500, block_sizes=[8, 64], budget_bp=[1500, 800], S=4, W=96,
                c_heavy=2.0, heavy_count=4, recency=300)
    base.update(kw)
    return synth.Workload(name, **base)


@pytest.mark.parametrize("mode", ["minmax", "mean"])
def test_ragged_batch_mixed_block_sizes(mode):
    # G = 3, block sizes 8 and 64, lengths not multiples of the page or block
    wl = _small(lens=[1500, 1013, 333])
    _full_pipeline(wl, 3, mode)


def test_short_and_empty_sequences():
    # L = 0 (empty: O = 0, lse = -inf), L < S, L < S + W (dense only), L = 1
    wl = _small(B=4, lens=[0, 3, 77, 1], L=100, heavy_count=0, recency=0)
    _full_pipeline(wl, 4, "minmax")


def test_full_budget_is_dense_attention():
    wl = _small(B=2, lens=[1500, 999])
    ks = []
    for h in range(wl.Hq):
        j0, j1 = orc.candidate_blocks(1500, wl.S, wl.W, wl.block_sizes[h // wl.G])
        ks.append(j1 - j0)
    prob, dev, ws, nc, ref_sel = _full_pipeline(wl, 5, "minmax", ks=ks)
    # and equals plain softmax over [0, L)
    out, lse = H.gpu_decode(prob, dev, *H.gpu_select(prob, dev, H.gpu_summaries(prob, dev, ws), ws)[:2], ws)
    for b in range(wl.B):
        for h in range(wl.Hq):
            kseq, vseq = H.oracle_kv(nc, b, h // wl.G)
            L = int(nc.seq_lens[b])
            O, lz = orc.attend(nc.q[b, h], kseq, vseq, np.arange(L), prob.scale)
            H.assert_close(out[b, h].cpu().numpy(), O, "dense O")


def test_long_ragged_sequences_span_several_tile_windows():
    # more than 4096 pages a sequence: each window of 4096 pages (65536
    # tokens) gets its own tile-list segment and builder CTA.  The lengths end
    # inside window 2, exactly on the window 0/1 edge, inside window 1 with
    # window 2 empty, and at 0 (no tile at all: O = 0, lse = -inf).
    wl = _small("long_ragged", B=4, L=150000, lens=[150000, 65536, 70001, 0], block_sizes=[16, 64],
                budget_bp=[500, 500], W=1024, heavy_count=6, recency=2000)
    _full_pipeline(wl, 7, "minmax")


def test_token_selections_on_long_ragged_sequences():
    # token granularity through sa_sparse_decode across tile-list windows:
    # per head a seeded set of tokens of the middle region (some repeated,
    # some outside it, which must be ignored)
    wl = _small("long_ragged", B=3, L=150000, lens=[150000, 70001, 0], block_sizes=[16, 64],
                budget_bp=[500, 500], W=1024, heavy_count=6, recency=2000)
    case = synth.make_decode_case(wl, 8)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    kcap = 1200
    prob = H.make_problem(wl, ks, kcap=kcap)
    rng = np.random.default_rng(8)
    sel, ref_sel = {}, {}
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        for h in range(wl.Hq):
            s_end, w_beg = min(L, wl.S), max(L - wl.W, min(L, wl.S))
            toks = np.sort(rng.choice(np.arange(s_end, w_beg), size=min(1000, max(0, w_beg - s_end)), replace=False)) \
                if w_beg > s_end else np.zeros(0, np.int64)
            ref_sel[(b, h)] = toks
            extra = list(toks[:50]) + [L + 5, -1]   # repeats and entries outside the middle region
            sel[(b, h)] = np.array(list(toks) + extra, dtype=np.int64)
    idx, cnt = H.sel_to_tensor(prob, sel)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    out, lse = H.gpu_decode(prob, dev, idx, cnt, ws, gran=sa.SEL_TOKEN)
    ref = H.oracle_decode(nc, wl, ref_sel, sa.SEL_TOKEN, prob.scale)
    _check_decode(out, lse, ref)
    assert ws.status() == sa.SA_OK


def test_zero_budget_is_dense_part_only():
    wl = _small(B=2)
    _full_pipeline(wl, 6, "mean", ks=[0] * wl.Hq)


def test_decode_given_oracle_index_sets_with_duplicates():
    # the decode step alone, fed the oracle's selection plus duplicates and
    # entries outside M (which must be ignored)
    wl = _small(B=2, lens=[1500, 1200])
    case = synth.make_decode_case(wl, 7)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    kcap = max(ks) * 2 + 4
    prob = H.make_problem(wl, ks, kcap=kcap)
    ref_sel = H.oracle_select(nc, wl, ks, "minmax")
    sel = {}
    for (b, h), (s, ids, _) in ref_sel.items():
        extra = [int(s[0])] if len(s) else []
        big = 10 ** 6
        sel[(b, h)] = np.array(list(s) + extra + [-3, big], dtype=np.int64)
    idx, cnt = H.sel_to_tensor(prob, sel)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    out, lse = H.gpu_decode(prob, dev, idx, cnt, ws)
    ref = H.oracle_decode(nc, wl, {k: v[0] for k, v in ref_sel.items()}, sa.SEL_BLOCK, prob.scale)
    _check_decode(out, lse, ref)


def test_token_granularity_and_logits():
    wl = _small(B=2, lens=[1500, 700])
    case = synth.make_decode_case(wl, 8)
    nc = H.to_np_case(case)
    rng = np.random.default_rng(8)
    kcap = 300
    prob = H.make_problem(wl, [0] * wl.Hq, kcap=kcap)
    sel = {}
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        for h in range(wl.Hq):
            n = int(rng.integers(0, 250))
            t = np.sort(rng.integers(0, L, n))
            sel[(b, h)] = t
    idx, cnt = H.sel_to_tensor(prob, sel)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    logits = torch.full((wl.B, wl.Hq, prob.max_pages_per_seq * 16), float("nan"), device="cuda")
    out, lse = H.gpu_decode(prob, dev, idx, cnt, ws, gran=sa.SEL_TOKEN, logits=logits)
    ref = H.oracle_decode(nc, wl, sel, sa.SEL_TOKEN, prob.scale)
    _check_decode(out, lse, ref)
    lg = logits.cpu().numpy()
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        s_end, w_beg = orc.partition(L, wl.S, wl.W)
        for h in range(wl.Hq):
            kseq, _ = H.oracle_kv(nc, b, h // wl.G)
            toks = np.array(sorted(set(orc.dense_tokens(L, wl.S, wl.W).tolist()) |
                                   set(int(t) for t in sel[(b, h)] if s_end <= t < w_beg)))
            zr = orc.attention_logits(nc.q[b, h], kseq, toks, prob.scale)
            H.assert_close(lg[b, h, toks], zr, "logits")
            others = np.setdiff1d(np.arange(lg.shape[2]), toks)
            assert np.all(np.isnan(lg[b, h, others])), "logits written outside the attended set"


def test_tail_summary_refresh_touches_only_last_block():
    wl = _small(B=2, lens=[1500, 1010])
    case = synth.make_decode_case(wl, 9)
    nc = H.to_np_case(case)
    prob = H.make_problem(wl, synth.k_per_qhead(wl), mode="mean")
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = torch.full(prob.summary_shape(), 7.0, dtype=torch.bfloat16, device="cuda")
    sa.block_summarize(prob, dev["k_pool"], dev["page_table"], dev["seq_lens"], summ, ws,
                       block_begin=sa.BLOCKS_TAIL)
    sg = summ.float().cpu().numpy()
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        for kvh in range(wl.Hk):
            Bs = wl.block_sizes[kvh]
            last = (L - 1) // Bs
            ref = H.oracle_summaries(nc, wl, b, kvh, "mean", last, last + 1)
            assert np.array_equal(sg[b, kvh, last], ref[0])
            assert np.all(sg[b, kvh, :last] == 7.0) and np.all(sg[b, kvh, last + 1:] == 7.0)


def test_bad_page_sets_status_without_fault():
    # a page-table entry outside the pool: the kernels skip that page and
    # report SA_ERR_BAD_PAGE through the status word; nothing traps
    wl = _small(B=2, heavy_count=2)
    case = synth.make_decode_case(wl, 10)
    prob = H.make_problem(wl, [0] * wl.Hq, kcap=4)
    dev = H.to_dev(case)
    dev["page_table"][1, 3] = prob.num_pages + 5
    ws = sa.Workspace(prob)
    H.gpu_summaries(prob, dev, ws)
    assert ws.status() == sa.SA_ERR_BAD_PAGE
    assert ws.status() == sa.SA_OK            # reading clears it
    sel = {(b, h): np.array([3 * 16 + 5]) for b in range(wl.B) for h in range(wl.Hq)}
    idx, cnt = H.sel_to_tensor(prob, sel)
    out, lse = H.gpu_decode(prob, dev, idx, cnt, ws, gran=sa.SEL_TOKEN)
    assert ws.status() == sa.SA_ERR_BAD_PAGE
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()


def test_lse_merge_standalone():
    rng = np.random.default_rng(11)
    n, D = 1000, 128
    oa = rng.standard_normal((n, D)).astype(np.float32)
    ob = rng.standard_normal((n, D)).astype(np.float32)
    la = (rng.standard_normal(n) * 5).astype(np.float32)
    lb = (rng.standard_normal(n) * 5).astype(np.float32)
    la[:10] = -np.inf
    lb[5:15] = -np.inf
    ref_o, ref_l = orc.lse_merge(oa, la, ob, lb)
    t = lambda x: torch.from_numpy(x).cuda()
    o = torch.empty(n, D, device="cuda")
    l = torch.empty(n, device="cuda")
    sa.lse_merge(t(oa), t(la), t(ob), t(lb), o, l)
    H.assert_close(o.cpu().numpy(), ref_o, "merge O")
    H.assert_close(l.cpu().numpy(), ref_l, "merge lse")


def test_repeated_calls_reuse_workspace():
    # split-K counters are left at zero: a second call gives the same result
    # (within rounding: tiles are consumed in the order they land)
    wl = synth.workload("tiny_4k")
    case = synth.make_decode_case(wl, 12)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    idx, cnt, _ = H.gpu_select(prob, dev, summ, ws)
    o1, l1 = H.gpu_decode(prob, dev, idx, cnt, ws)
    o2, l2 = H.gpu_decode(prob, dev, idx, cnt, ws)
    H.assert_close(o2.cpu().numpy(), o1.cpu().numpy(), "O, second call")
    H.assert_close(l2.cpu().numpy(), l1.cpu().numpy(), "lse, second call")


@pytest.mark.parametrize("name", ["tiny_4k", "llama_32k", "ragged"])
def test_decode_step_matches_separate_calls(name):
    # sa_decode_step = tail summary refresh + select_topk + sparse_decode
    if name == "ragged":
        wl = _small(lens=[1500, 1013, 333])
    else:
        wl = synth.workload(name)
    case = synth.make_decode_case(wl, 31)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    # poison the tail blocks so the refresh is checked too
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        for kvh in range(wl.Hk):
            if L > 0:
                summ[b, kvh, (L - 1) // wl.block_sizes[kvh]] = 3.0
    summ_ref = summ.clone()
    sa.block_summarize(prob, dev["k_pool"], dev["page_table"], dev["seq_lens"], summ_ref, ws,
                       block_begin=sa.BLOCKS_TAIL)
    idx_ref, cnt_ref, _ = H.gpu_select(prob, dev, summ_ref, ws, with_scores=False)
    o_ref, l_ref = H.gpu_decode(prob, dev, idx_ref, cnt_ref, ws)
    idx = torch.full_like(idx_ref, -5)
    cnt = torch.full_like(cnt_ref, -5)
    out = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(l_ref, float("nan"))
    sa.decode_step(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ, idx, cnt,
                   out, lse, ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    assert torch.equal(summ.view(torch.int16), summ_ref.view(torch.int16))
    assert torch.equal(cnt, cnt_ref)
    for b in range(wl.B):
        for h in range(wl.Hq):
            n = int(cnt_ref[b, h])
            assert torch.equal(idx[b, h, :n], idx_ref[b, h, :n])
    H.assert_close(out.cpu().numpy(), o_ref.cpu().numpy(), "step O")
    H.assert_close(lse.cpu().numpy(), l_ref.cpu().numpy(), "step lse")


@pytest.mark.gpu
def test_prepared_step_call_matches_decode_step():
    # sa.DecodeStepCall marshals once and passes only the stream on each call;
    # with fresh contents in the same buffers it gives decode_step's results
    wl = synth.workload("tiny_4k")
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    ws = sa.Workspace(prob)
    case = synth.make_decode_case(wl, 41)
    dev = H.to_dev(case)
    summ = H.gpu_summaries(prob, dev, ws)
    idx = torch.empty(wl.B, wl.Hq, prob.kcap, dtype=torch.int32, device="cuda")
    cnt = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.float32, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device="cuda")
    call = sa.DecodeStepCall(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ,
                             idx, cnt, out, lse, ws)
    for seed in (42, 43):
        q_new = synth.make_decode_case(wl, seed).q.to("cuda")
        dev["q"].copy_(q_new)
        call()
        o1, l1, i1, c1 = out.clone(), lse.clone(), idx.clone(), cnt.clone()
        sa.decode_step(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ, idx,
                       cnt, out, lse, ws)
        torch.cuda.synchronize()
        assert ws.status() == sa.SA_OK
        assert torch.equal(c1, cnt) and torch.equal(i1, idx)
        H.assert_close(o1.cpu().numpy(), out.cpu().numpy(), "prepared O")
        H.assert_close(l1.cpu().numpy(), lse.cpu().numpy(), "prepared lse")


@pytest.mark.parametrize("G", [1, 2, 5, 6, 8])
def test_group_sizes(G):
    # every group size the kernels are instantiated for beyond 3, 4 and 7 (8 is the largest)
    wl = _small(name=f"g{G}", B=2, Hq=2 * G, Hk=2, block_sizes=[16, 32], budget_bp=[1000, 700],
                lens=[1500, 1111])
    prob, dev, ws, nc, ref_sel = _full_pipeline(wl, 5 + G, "minmax")
    # the fused step (scores, top-k + tiles + tail summary, decode, merge) on fresh summaries
    summ = H.gpu_summaries(prob, dev, ws)
    idx = torch.full((wl.B, wl.Hq, prob.kcap), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((wl.B, wl.Hq), -5, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    sa.decode_step(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ, idx, cnt,
                   out, lse, ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    _check_selection(prob, wl, nc, idx, cnt, None, ref_sel)
    ref_dec = H.oracle_decode(nc, wl, {k: v[0] for k, v in ref_sel.items()}, sa.SEL_BLOCK, prob.scale)
    _check_decode(out, lse, ref_dec)
