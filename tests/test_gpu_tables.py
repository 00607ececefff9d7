"""Score-table driven selection over consecutive decode steps, teacher-forced
against the oracle:
  1. given the GPU's updated fp32 tables, the oracle's threshold + expansion
     reproduces the GPU's candidate list bit for bit;
  2. given the GPU's input tables and the previous step's candidate list, the
     oracle's fp64 update matches the GPU's tables within 1e-6 + 1e-4 |T|;
  3. given the candidate list, O and lse are within the parity tolerance."""
import math

import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _run(wl, seed, nsteps, heads=None):
    case = synth.make_table_case(wl, seed)
    B, Hq, Hk, G = wl.B, wl.Hq, wl.Hk, wl.G
    mpp = wl.max_pages_per_seq
    N = mpp * wl.P
    prob = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                      block_sizes=[16] * Hk, k_per_head=[0] * Hq, kcap=wl.kcap)
    ws = sa.Workspace(prob)
    kp, vp, pt = case.k_pool.cuda(), case.v_pool.cuda(), case.page_table.cuda()
    kp_np, vp_np, pt_np = orc.to_np(case.k_pool), orc.to_np(case.v_pool), orc.to_np(case.page_table)
    tv = [case.vert0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    ts = [case.slash0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    cand = [torch.zeros(B, Hq, wl.kcap, dtype=torch.int32, device="cuda") for _ in range(2)]
    cnt = [torch.zeros(B, Hq, dtype=torch.int32, device="cuda") for _ in range(2)]
    logits = torch.zeros(B, Hq, N, device="cuda")
    heads = heads or [(b, h) for b in range(B) for h in range(Hq)]
    prev = None
    prev_L = None
    n_cands = []
    for t in range(nsteps):
        L = wl.L0 + t
        seq_lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
        cur, nxt = t % 2, (t + 1) % 2
        sa.update_score_tables(prob, tv[cur], ts[cur], tv[nxt], ts[nxt], seq_lens, cand[cur], cnt[cur], ws,
                               beta=wl.beta, prev=prev)
        torch.cuda.synchronize()
        assert ws.status() == sa.SA_OK
        v_in, s_in = tv[cur].cpu().numpy(), ts[cur].cpu().numpy()
        v_out, s_out = tv[nxt].cpu().numpy(), ts[nxt].cpu().numpy()
        c_gpu, n_gpu = cand[cur].cpu().numpy(), cnt[cur].cpu().numpy()
        for (b, h) in heads:
            # 1. selection from the GPU's tables, bit for bit
            c_ref, over = orc.table_candidates(v_out[b, h], s_out[b, h], L, wl.S, wl.W, wl.beta, wl.kcap)
            assert not over
            assert np.array_equal(c_gpu[b, h, :n_gpu[b, h]], c_ref), f"step {t} (b={b}, h={h}) candidates differ"
            # 2. the update, from the GPU's input tables and the previous candidates
            if prev is not None:
                kseq = orc.gather_sequence(kp_np, pt_np[b], h // G, prev_L)
                q_prev = orc.to_np(case.q_steps[t - 1, b, h])
                pos, w = orc.merged_weights(q_prev, kseq, prev_L, wl.S, wl.W,
                                            prev_c[b, h, :prev_n[b, h]], prob.scale)
                v_ref, s_ref = orc.table_update(v_in[b, h].astype(np.float64), s_in[b, h].astype(np.float64),
                                                prev_L, pos, w)
            else:
                v_ref, s_ref = v_in[b, h], s_in[b, h]
            for got, ref, nm in ((v_out[b, h], v_ref, "vertical"), (s_out[b, h], s_ref, "slash")):
                err = np.abs(got.astype(np.float64) - ref)
                assert np.all(err <= 1e-6 + 1e-4 * np.abs(ref)), f"step {t} {nm} table: max err {err.max():.3e}"
        n_cands.append(int(n_gpu.mean()))
        # 3. decode over I + the candidate tokens, with logits for the next update
        q = case.q_steps[t].cuda()
        dev = dict(q=q, k_pool=kp, v_pool=vp, page_table=pt, seq_lens=seq_lens)
        o, l = H.gpu_decode(prob, dev, cand[cur], cnt[cur], ws, gran=sa.SEL_TOKEN, logits=logits)
        o_np, l_np = o.cpu().numpy(), l.cpu().numpy()
        for (b, h) in heads[:: max(1, len(heads) // 16)]:
            kseq = orc.gather_sequence(kp_np, pt_np[b], h // G, L)
            vseq = orc.gather_sequence(vp_np, pt_np[b], h // G, L)
            qh = orc.to_np(case.q_steps[t, b, h])
            I = orc.dense_tokens(L, wl.S, wl.W)
            Jt = c_gpu[b, h, :n_gpu[b, h]]
            O_I, lI = orc.attend(qh, kseq, vseq, I, prob.scale)
            O_J, lJ = orc.attend(qh, kseq, vseq, Jt, prob.scale)
            O_ref, lse_ref = orc.lse_merge(O_I, lI, O_J, lJ)
            H.assert_close(o_np[b, h], O_ref, f"step {t} O")
            H.assert_close(np.array([l_np[b, h]]), np.array([float(lse_ref)]), f"step {t} lse")
        prev = dict(prev_seq_lens=seq_lens, prev_sel_idx=cand[cur], prev_sel_cnt=cnt[cur], prev_logits=logits,
                    prev_lse=l)
        prev_c, prev_n, prev_L = c_gpu, n_gpu, L
    return n_cands


def test_tables_small_all_steps():
    wl = synth.table_workload("tables_small")
    n = _run(wl, 0, wl.steps)
    assert min(n) > 0   # the planted entries keep producing candidates


def test_tables_128k_llama_shape_64_steps():
    # the 131072-token, batch-4 Llama-shaped workload at full size over all 64
    # steps (the GPU runs every head; the oracle checks a sample of heads)
    wl = synth.table_workload("tables_128k")
    heads = [(0, 0), (1, 9), (2, 17), (3, 31)]
    n = _run(wl, 3, wl.steps, heads=heads)
    assert min(n) > 0


def test_tables_small_free_running_overlap():
    """Free-running comparison (reported, not gated): the GPU path and the
    oracle each carry their own tables over all steps, and the candidate sets
    they pick are compared per step by Jaccard overlap.  exp() differs in the
    last bits between the two, so a weight near the threshold can flip a
    candidate and the runs drift apart; the teacher-forced tests above are the
    parity gate."""
    wl = synth.table_workload("tables_small")
    case = synth.make_table_case(wl, 5)
    B, Hq, Hk, G = wl.B, wl.Hq, wl.Hk, wl.G
    mpp = wl.max_pages_per_seq
    N = mpp * wl.P
    prob = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                      block_sizes=[16] * Hk, k_per_head=[0] * Hq, kcap=wl.kcap)
    ws = sa.Workspace(prob)
    kp, vp, pt = case.k_pool.cuda(), case.v_pool.cuda(), case.page_table.cuda()
    kp_np, vp_np, pt_np = orc.to_np(case.k_pool), orc.to_np(case.v_pool), orc.to_np(case.page_table)
    tv = [case.vert0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    ts = [case.slash0.cuda(), torch.empty(B, Hq, N, device="cuda")]
    cand = [torch.zeros(B, Hq, wl.kcap, dtype=torch.int32, device="cuda") for _ in range(2)]
    cnt = [torch.zeros(B, Hq, dtype=torch.int32, device="cuda") for _ in range(2)]
    logits = torch.zeros(B, Hq, N, device="cuda")
    ov = orc.to_np(case.vert0).astype(np.float64)
    osl = orc.to_np(case.slash0).astype(np.float64)
    prev = None
    o_prev = None
    jaccard = []
    for t in range(wl.steps):
        L = wl.L0 + t
        seq_lens = torch.full((B,), L, dtype=torch.int32, device="cuda")
        cur, nxt = t % 2, (t + 1) % 2
        sa.update_score_tables(prob, tv[cur], ts[cur], tv[nxt], ts[nxt], seq_lens, cand[cur], cnt[cur], ws,
                               beta=wl.beta, prev=prev)
        q = case.q_steps[t].cuda()
        dev = dict(q=q, k_pool=kp, v_pool=vp, page_table=pt, seq_lens=seq_lens)
        o, l = H.gpu_decode(prob, dev, cand[cur], cnt[cur], ws, gran=sa.SEL_TOKEN, logits=logits)
        torch.cuda.synchronize()
        assert ws.status() == sa.SA_OK
        c_gpu, n_gpu = cand[cur].cpu().numpy(), cnt[cur].cpu().numpy()
        step = []
        new_o = {}
        for b in range(B):
            for h in range(Hq):
                kseq = orc.gather_sequence(kp_np, pt_np[b], h // G, L)
                if o_prev is not None:   # the oracle's own update from its own previous step
                    qp, Lp, cp = o_prev[(b, h)]
                    pos, w = orc.merged_weights(qp, orc.gather_sequence(kp_np, pt_np[b], h // G, Lp), Lp, wl.S,
                                                wl.W, cp, prob.scale)
                    ov[b, h], osl[b, h] = orc.table_update(ov[b, h], osl[b, h], Lp, pos, w)
                c_ref, _ = orc.table_candidates(ov[b, h].astype(np.float32), osl[b, h].astype(np.float32), L,
                                                wl.S, wl.W, wl.beta, wl.kcap)
                a = set(c_gpu[b, h, :n_gpu[b, h]].tolist())
                r = set(c_ref.tolist())
                step.append(len(a & r) / max(1, len(a | r)))
                new_o[(b, h)] = (orc.to_np(case.q_steps[t, b, h]), L, c_ref)
        o_prev = new_o
        jaccard.append(float(np.mean(step)))
        prev = dict(prev_seq_lens=seq_lens, prev_sel_idx=cand[cur], prev_sel_cnt=cnt[cur], prev_logits=logits,
                    prev_lse=l)
    print("free-running Jaccard per step:", " ".join(f"{x:.3f}" for x in jaccard))
    assert len(jaccard) == wl.steps and all(0.0 <= x <= 1.0 for x in jaccard)
    assert jaccard[0] == 1.0   # step 0 starts from the same tables
