"""Cells of the throughput sweep of the full decode-attention stack (batch x
context x budget, one appended token per step) against the oracle: three
appending decode steps (sa_decode_step_append), then the last step's tail
summaries, selections and outputs on sampled (sequence, KV head) units.  The
100 % budget cell must equal dense attention over the whole context."""
import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu

STEPS = 3


def _run_cell(B, ctx, bp, units, seed=21):
    wl = synth.sweep_workload(B, ctx, bp)
    case = synth.make_decode_case(wl, seed)
    L_final = ctx + STEPS
    ks = synth.k_per_qhead(wl, L_final)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)            # the prefill's full build
    g = torch.Generator().manual_seed(seed + 7)
    kp, vp = dev["k_pool"], dev["v_pool"]
    idx = torch.empty(B, wl.Hq, prob.kcap, dtype=torch.int32, device="cuda")
    cnt = torch.empty(B, wl.Hq, dtype=torch.int32, device="cuda")
    out = torch.empty(B, wl.Hq, wl.D, device="cuda")
    lse = torch.empty(B, wl.Hq, device="cuda")
    new_rows = []
    for s in range(STEPS):
        lens = dev["seq_lens"] + (s + 1)
        k_new = torch.randn(B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
        v_new = torch.randn(B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
        q = torch.randn(B, wl.Hq, wl.D, generator=g).to(torch.bfloat16).cuda() if s + 1 < STEPS else dev["q"]
        sa.decode_step_append(prob, q, k_new, v_new, kp, vp, dev["page_table"], lens, summ, idx, cnt, out, lse, ws)
        new_rows.append((k_new.cpu(), v_new.cpu()))
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    # the oracle's pools: the synthetic ones with the appended rows written by indexing
    k_np, v_np = orc.to_np(case.k_pool).copy(), orc.to_np(case.v_pool).copy()
    pt = orc.to_np(case.page_table)
    for s, (kn, vn) in enumerate(new_rows):
        for b in range(B):
            t = ctx + s
            phys = int(pt[b, t // wl.P])
            k_np[phys, :, t % wl.P] = orc.to_np(kn[b])
            v_np[phys, :, t % wl.P] = orc.to_np(vn[b])
    nc = H.NpCase(q=orc.to_np(case.q), k_pool=k_np, v_pool=v_np, page_table=pt,
                  seq_lens=np.full(B, L_final, dtype=np.int64))
    sel = H.oracle_select(nc, wl, ks, "minmax", units)
    idx_np, cnt_np = idx.cpu().numpy(), cnt.cpu().numpy()
    for (b, h), (s_ref, _, _) in sel.items():
        assert np.array_equal(idx_np[b, h, :cnt_np[b, h]], s_ref), f"selection (b={b}, h={h})"
    dec = H.oracle_decode(nc, wl, {k: v[0] for k, v in sel.items()}, sa.SEL_BLOCK, prob.scale, units)
    o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), (O, l) in dec.items():
        H.assert_close(o_np[b, h], O, f"O (b={b}, h={h})")
        H.assert_close(np.array([l_np[b, h]]), np.array([l]), f"lse (b={b}, h={h})")
    # the blocks the appended tokens landed in: summaries refreshed by the steps
    summ_np = summ.float().cpu().numpy()
    for b, kvh in units:
        kseq, _ = H.oracle_kv(nc, b, kvh)
        for j in sorted({(ctx + s) // 16 for s in range(STEPS)}):
            ref = orc.summarize_sequence(kseq, 16, "minmax", j, j + 1)[0]
            assert np.array_equal(summ_np[b, kvh, j].reshape(ref.shape), ref), f"tail summary (b={b}, kvh={kvh}, j={j})"
    return wl, prob, nc, sel, dec


@pytest.mark.parametrize("B,ctx,bp,units", [
    (1, 8192, 100, [(0, 0), (0, 7)]),                  # 1 % budget
    (4, 32768, 1000, [(0, 2), (3, 5)]),                # 10 %
    (64, 8192, 500, [(0, 1), (37, 4), (63, 7)]),       # batch 64
    (1, 262144, 500, [(0, 3)]),                        # 256K context
])
def test_sweep_cell(B, ctx, bp, units):
    _run_cell(B, ctx, bp, units)


def test_sweep_cell_dense_budget_is_dense_attention():
    B, ctx = 16, 8192
    wl, prob, nc, sel, dec = _run_cell(B, ctx, 10000, [(0, 0), (15, 6)])
    L = ctx + STEPS
    for (b, h), (O, l) in dec.items():
        s_ref = sel[(b, h)][0]
        j0, j1 = orc.candidate_blocks(L, wl.S, wl.W, 16)
        assert np.array_equal(s_ref, np.arange(j0, j1))     # every candidate kept
        kseq, vseq = H.oracle_kv(nc, b, h // wl.G)
        Od, ld = orc.attend(nc.q[b, h], kseq, vseq, np.arange(L), prob.scale)
        assert np.abs(O - Od).max() < 1e-9 and abs(l - ld) < 1e-9
