"""Exact top-k inside the score-table candidates (sa_select_tokens) against
the oracle: kept positions and every candidate's score bit for bit, and the
decode over the kept tokens within the parity tolerance."""
import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _run(name, k_tok, heads=None, seed=4):
    wl = synth.table_workload(name)
    case = synth.make_table_case(wl, seed)
    B, Hq, Hk, G = wl.B, wl.Hq, wl.Hk, wl.G
    mpp = wl.max_pages_per_seq
    N = mpp * wl.P
    prob = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                      block_sizes=[16] * Hk, k_per_head=[k_tok] * Hq, kcap=wl.kcap)
    ws = sa.Workspace(prob)
    kp, vp, pt = case.k_pool.cuda(), case.v_pool.cuda(), case.page_table.cuda()
    kp_np, vp_np, pt_np = orc.to_np(case.k_pool), orc.to_np(case.v_pool), orc.to_np(case.page_table)
    L = wl.L0
    seq_lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
    tv = [case.vert0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    ts = [case.slash0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    cand = torch.zeros(B, Hq, wl.kcap, dtype=torch.int32, device="cuda")
    ccnt = torch.zeros(B, Hq, dtype=torch.int32, device="cuda")
    sa.update_score_tables(prob, tv[0], ts[0], tv[1], ts[1], seq_lens, cand, ccnt, ws, beta=wl.beta)
    q = case.q_steps[0].cuda()
    sel = torch.full((B, Hq, wl.kcap), -3, dtype=torch.int32, device="cuda")
    scnt = torch.full((B, Hq), -3, dtype=torch.int32, device="cuda")
    scores = torch.full((B, Hq, wl.kcap), float("nan"), device="cuda")
    sa.select_tokens(prob, q, kp, pt, seq_lens, cand, ccnt, sel, scnt, ws, scores=scores)
    dev = dict(q=q, k_pool=kp, v_pool=vp, page_table=pt, seq_lens=seq_lens)
    o, l = H.gpu_decode(prob, dev, sel, scnt, ws, gran=sa.SEL_TOKEN)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    c_np, cc_np = cand.cpu().numpy(), ccnt.cpu().numpy()
    s_np, sc_np, scores_np = sel.cpu().numpy(), scnt.cpu().numpy(), scores.cpu().numpy()
    o_np, l_np = o.cpu().numpy(), l.cpu().numpy()
    heads = heads or [(b, h) for b in range(B) for h in range(Hq)]
    for (b, h) in heads:
        kseq = orc.gather_sequence(kp_np, pt_np[b], h // G, L)
        qh = orc.to_np(case.q_steps[0, b, h])
        cands = c_np[b, h, :cc_np[b, h]]
        kept, sc = orc.exact_token_topk(qh, kseq, cands, k_tok)
        assert sc_np[b, h] == len(kept)
        assert np.array_equal(s_np[b, h, :sc_np[b, h]], kept), f"(b={b}, h={h}) kept tokens differ"
        assert np.array_equal(scores_np[b, h, :len(cands)].view(np.int32), sc.view(np.int32)), \
            f"(b={b}, h={h}) candidate scores differ"
        vseq = orc.gather_sequence(vp_np, pt_np[b], h // G, L)
        I = orc.dense_tokens(L, wl.S, wl.W)
        O_I, lI = orc.attend(qh, kseq, vseq, I, prob.scale)
        O_J, lJ = orc.attend(qh, kseq, vseq, kept, prob.scale)
        O_ref, lse_ref = orc.lse_merge(O_I, lI, O_J, lJ)
        H.assert_close(o_np[b, h], O_ref, f"(b={b}, h={h}) O")
        H.assert_close(np.array([l_np[b, h]]), np.array([float(lse_ref)]), f"(b={b}, h={h}) lse")
    return cc_np


@pytest.mark.parametrize("k_tok", [0, 1, 5, 512])
def test_exact_token_topk_tables_small(k_tok):
    # 512 = kcap of the workload: every candidate is kept
    cc = _run("tables_small", k_tok)
    assert cc.max() > 5   # enough candidates for the small budgets to choose


def test_exact_token_topk_tables_128k_sampled_heads():
    _run("tables_128k", 8, heads=[(0, 0), (1, 13), (2, 22), (3, 31)])
