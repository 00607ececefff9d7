"""Head-sparsity bypass (LFPS Algorithm 1 step 1, Eq. (5), Eq. (6), App. B.1)
against the oracle: the running KV sums, the sink share rho and the bypass
decision per head, the bypass output (mean value row, estimated lse), the
decode step that leaves bypassed heads out, and the frozen score tables.

rho is fp32 on the GPU and fp64 in the oracle: it is compared within 1e-4,
and the decision (rho > eps, taken by the GPU in fp32) must equal the
oracle's wherever the oracle's rho is further than that from eps."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu

EPS = orc.BYPASS_EPS
RHO_TOL = 1e-4


def _setup(name, seed=5, extra_tokens=0):
    wl = synth.workload(name)
    if extra_tokens:
        wl = dataclasses.replace(wl, extra_tokens=extra_tokens)
    case = synth.make_decode_case(wl, seed)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    return wl, case, ks, prob, H.to_dev(case), sa.Workspace(prob)


def _gpu_stats(prob, dev, ws):
    st = torch.full(sa.kv_stats_shape(prob), float("nan"), device="cuda")
    sa.kv_stats(prob, dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], st, ws)
    return st


def _check_stats(st, nc, units):
    st_np = st.cpu().numpy().astype(np.float64)
    for b, kvh in units:
        sums, mags = H.oracle_kv_stats(nc, b, kvh)
        err = np.abs(st_np[b, kvh] - sums)
        assert (err <= 4e-5 * mags + 1e-6).all(), f"kv sums (b={b}, kvh={kvh}) max err {err.max()}"


def _check_estimate(ref, rho, byp, out, lse, untouched_sentinel=True):
    """rho / decisions / bypass outputs against the oracle; rows not bypassed
    must still hold the NaN sentinel when untouched_sentinel."""
    rho_np, byp_np = rho.cpu().numpy(), byp.cpu().numpy()
    o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
    n_by = 0
    for (b, h), (r_ref, lse_ref, vbar) in ref.items():
        assert abs(float(rho_np[b, h]) - r_ref) <= RHO_TOL, f"rho (b={b}, h={h}) {rho_np[b, h]} vs {r_ref}"
        assert byp_np[b, h] == int(float(rho_np[b, h]) > EPS), f"flag (b={b}, h={h}) not rho > eps"
        if abs(r_ref - EPS) > RHO_TOL:
            assert byp_np[b, h] == int(orc.is_bypassed(r_ref)), f"decision (b={b}, h={h})"
        if byp_np[b, h]:
            n_by += 1
            H.assert_close(o_np[b, h], vbar, f"bypass O (b={b}, h={h})")
            H.assert_close(np.array([l_np[b, h]]), np.array([lse_ref]), f"bypass lse (b={b}, h={h})")
        elif untouched_sentinel:
            assert np.isnan(o_np[b, h]).all() and np.isnan(l_np[b, h]), f"row (b={b}, h={h}) written"
    return n_by


@pytest.mark.parametrize("name,units", [
    ("tiny_4k_sinkheads", None),
    ("llama_32k_sinkheads", [(0, 0), (0, 1), (1, 2), (3, 6)]),   # seed 5 plants heads in the last three
])
def test_kv_stats_and_head_sparsity(name, units):
    wl, case, ks, prob, dev, ws = _setup(name)
    nc = H.to_np_case(case)
    units = units or [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    st = _gpu_stats(prob, dev, ws)
    rho = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    byp = torch.full((wl.B, wl.Hq), -1, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    sa.head_sparsity(prob, dev["q"], dev["k_pool"], dev["page_table"], dev["seq_lens"], st, byp, out, lse, ws,
                     eps=EPS, rho=rho)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    _check_stats(st, nc, units)
    ref = H.oracle_bypass(nc, wl, prob.scale, units)
    n_by = _check_estimate(ref, rho, byp, out, lse)
    assert 0 < n_by < len(units) * wl.G   # both kinds of head are there


def _oracle_step(nc, wl, ks, prob, units):
    """Expected (bypass estimate, selections, decode) of the bypass step."""
    est = H.oracle_bypass(nc, wl, prob.scale, units)
    sel = H.oracle_select(nc, wl, ks, "minmax", units)
    dec = H.oracle_decode(nc, wl, {k: v[0] for k, v in sel.items()}, sa.SEL_BLOCK, prob.scale, units)
    return est, sel, dec


def _check_step(est, sel, dec, rho, byp, idx, cnt, out, lse):
    _check_estimate(est, rho, byp, out, lse, untouched_sentinel=False)
    byp_np, idx_np, cnt_np = byp.cpu().numpy(), idx.cpu().numpy(), cnt.cpu().numpy()
    o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), (s_ref, _, _) in sel.items():
        if byp_np[b, h]:
            assert cnt_np[b, h] == 0, f"bypassed head (b={b}, h={h}) selected blocks"
            continue
        assert np.array_equal(idx_np[b, h, :cnt_np[b, h]], s_ref), f"selection (b={b}, h={h})"
        O, l = dec[(b, h)]
        H.assert_close(o_np[b, h], O, f"step O (b={b}, h={h})")
        H.assert_close(np.array([l_np[b, h]]), np.array([l]), f"step lse (b={b}, h={h})")


@pytest.mark.parametrize("name,units", [
    ("tiny_4k_sinkheads", None),
    ("llama_32k_sinkheads", [(0, 3), (1, 7), (2, 4)]),   # each holds a planted head (seed 5)
])
def test_decode_step_bypass_matches_oracle(name, units):
    wl, case, ks, prob, dev, ws = _setup(name)
    nc = H.to_np_case(case)
    units = units or [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    summ = H.gpu_summaries(prob, dev, ws)
    st = _gpu_stats(prob, dev, ws)
    rho = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    byp = torch.full((wl.B, wl.Hq), -1, dtype=torch.int32, device="cuda")
    idx = torch.full((wl.B, wl.Hq, prob.kcap), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((wl.B, wl.Hq), -5, dtype=torch.int32, device="cuda")
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    sa.decode_step_bypass(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ,
                          st, idx, cnt, out, lse, byp, ws, eps=EPS, rho=rho)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    _check_step(*_oracle_step(nc, wl, ks, prob, units), rho, byp, idx, cnt, out, lse)
    if name == "tiny_4k_sinkheads":
        # the one-token sequence: every head bypassed, and the bypass output is exact attention
        assert byp[3].cpu().numpy().tolist() == [1] * wl.Hq


def test_decode_step_bypass_with_append():
    wl, case, ks, prob, dev, ws = _setup("tiny_4k_sinkheads", seed=6, extra_tokens=16)
    st = _gpu_stats(prob, dev, ws)                 # the L tokens before the new one
    summ = H.gpu_summaries(prob, dev, ws)
    g = torch.Generator().manual_seed(61)
    k_new = torch.randn(wl.B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn(wl.B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
    lens1 = dev["seq_lens"] + 1
    kp, vp = dev["k_pool"].clone(), dev["v_pool"].clone()
    rho = torch.empty(wl.B, wl.Hq, device="cuda")
    byp = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    idx = torch.empty(wl.B, wl.Hq, prob.kcap, dtype=torch.int32, device="cuda")
    cnt = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    out = torch.empty(wl.B, wl.Hq, wl.D, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    sa.decode_step_bypass(prob, dev["q"], kp, vp, dev["page_table"], lens1, summ, st, idx, cnt, out, lse, byp, ws,
                          eps=EPS, rho=rho, k_new=k_new, v_new=v_new)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    # the oracle sees the pools with the new rows written by indexing
    kr, vr = dev["k_pool"].clone(), dev["v_pool"].clone()
    pt = dev["page_table"].cpu()
    for b in range(wl.B):
        t = int(lens1[b]) - 1
        phys = int(pt[b, t // wl.P])
        kr[phys, :, t % wl.P] = k_new[b]
        vr[phys, :, t % wl.P] = v_new[b]
    assert torch.equal(kp.view(torch.int16), kr.view(torch.int16))
    assert torch.equal(vp.view(torch.int16), vr.view(torch.int16))
    nc = H.NpCase(q=orc.to_np(case.q), k_pool=orc.to_np(kr.cpu()), v_pool=orc.to_np(vr.cpu()),
                  page_table=orc.to_np(case.page_table), seq_lens=orc.to_np(lens1.cpu()))
    units = [(b, kvh) for b in range(wl.B) for kvh in range(wl.Hk)]
    _check_stats(st, nc, units)                    # the sums now include the new rows
    _check_step(*_oracle_step(nc, wl, ks, prob, units), rho, byp, idx, cnt, out, lse)


def test_sparse_decode_leaves_bypassed_heads_out():
    wl, case, ks, prob, dev, ws = _setup("tiny_4k_sinkheads")
    nc = H.to_np_case(case)
    st = _gpu_stats(prob, dev, ws)
    summ = H.gpu_summaries(prob, dev, ws)
    idx, cnt, _ = H.gpu_select(prob, dev, summ, ws, with_scores=False)
    byp = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    rho = torch.empty(wl.B, wl.Hq, device="cuda")
    out = torch.full((wl.B, wl.Hq, wl.D), float("nan"), device="cuda")
    lse = torch.full((wl.B, wl.Hq), float("nan"), device="cuda")
    sa.head_sparsity(prob, dev["q"], dev["k_pool"], dev["page_table"], dev["seq_lens"], st, byp, out, lse, ws,
                     rho=rho)
    sa.sparse_decode(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], idx, cnt, out,
                     lse, ws, bypass=byp)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    est, sel, dec = _oracle_step(nc, wl, ks, prob, None)
    _check_estimate(est, rho, byp, out, lse, untouched_sentinel=False)
    byp_np, o_np, l_np = byp.cpu().numpy(), out.cpu().numpy(), lse.cpu().numpy()
    assert byp_np.sum() > 0 and (byp_np == 0).sum() > 0
    for (b, h), (O, l) in dec.items():
        if not byp_np[b, h]:
            H.assert_close(o_np[b, h], O, f"O (b={b}, h={h})")
            H.assert_close(np.array([l_np[b, h]]), np.array([l]), f"lse (b={b}, h={h})")


def test_tables_of_bypassed_heads_are_frozen():
    wl = synth.table_workload("tables_small")
    case = synth.make_table_case(wl, 3)
    B, Hq, Hk = wl.B, wl.Hq, wl.Hk
    mpp = wl.max_pages_per_seq
    N = mpp * wl.P
    prob = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                      block_sizes=[16] * Hk, k_per_head=[8] * Hq, kcap=wl.kcap)
    ws = sa.Workspace(prob)
    L0 = wl.L0
    lens0 = torch.full((B,), L0, dtype=torch.int32, device="cuda")
    lens1 = lens0 + 1
    g = torch.Generator().manual_seed(9)
    logits = (torch.randn(B, Hq, N, generator=g) * 2).cuda()
    lse_prev = torch.logsumexp(logits[:, :, :L0], dim=-1).contiguous()
    sel = torch.stack([torch.stack([torch.sort(torch.randperm(L0 - wl.W - wl.S, generator=g)[:wl.kcap] + wl.S)[0]
                                    for _ in range(Hq)]) for _ in range(B)]).to(torch.int32).cuda()
    scnt = torch.full((B, Hq), min(40, wl.kcap), dtype=torch.int32, device="cuda")
    prev = dict(prev_seq_lens=lens0, prev_sel_idx=sel, prev_sel_cnt=scnt, prev_logits=logits, prev_lse=lse_prev)
    frozen = (torch.rand(B, Hq, generator=g) < 0.3).to(torch.int32).cuda()
    frozen[0, 0], frozen[0, 1] = 1, 0
    vin, sin = case.vert0.cuda(), case.slash0.cuda()
    res = []
    for fl in (None, frozen):
        vo, so = torch.empty(B, Hq, N, device="cuda"), torch.empty(B, Hq, N, device="cuda")
        cand = torch.zeros(B, Hq, wl.kcap, dtype=torch.int32, device="cuda")
        ccnt = torch.zeros(B, Hq, dtype=torch.int32, device="cuda")
        sa.update_score_tables(prob, vin, sin, vo, so, lens1, cand, ccnt, ws, beta=wl.beta, prev=prev,
                               prev_bypass=fl)
        res.append((vo, so))
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    f = frozen.bool()
    (v_free, s_free), (v_fr, s_fr) = res
    assert torch.equal(v_fr[f], vin[f]) and torch.equal(s_fr[f], sin[f])          # copied unchanged
    assert torch.equal(v_fr[~f], v_free[~f]) and torch.equal(s_fr[~f], s_free[~f])  # others as without flags
    assert not torch.equal(v_free[f], vin[f])                                      # the update does change them
