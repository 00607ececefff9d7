"""Group-shared selection (SA_SELECT_GROUP): every query head of a KV head
keeps the blocks ranked best by the fp32 sum of the group's canonical scores.
Selections are compared with the oracle bit for bit; the decode over them
within the parity tolerance."""
import numpy as np
import pytest
import torch

from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _check_selection(name, mode, units=None, seed=11):
    wl = synth.workload(name)
    case = synth.make_decode_case(wl, seed)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks, mode=mode, selection=sa.SELECT_GROUP)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    idx, cnt, _ = H.gpu_select(prob, dev, summ, ws, with_scores=False)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    ref = H.oracle_select_group(nc, wl, ks, mode, units)
    idx_np, cnt_np = idx.cpu().numpy(), cnt.cpu().numpy()
    for (b, h), (sel, _, _) in ref.items():
        got = idx_np[b, h, :cnt_np[b, h]]
        assert np.array_equal(got, sel), f"{name} {mode} (b={b}, h={h}) group selection differs"
    return wl, prob, dev, ws, summ, ks, nc, idx, cnt


@pytest.mark.parametrize("mode", ["minmax", "mean"])
def test_group_selection_tiny_4k(mode):
    _check_selection("tiny_4k", mode)


def test_group_selection_llama_32k_sampled_units():
    units = [(0, 0), (3, 5), (7, 7)]
    _check_selection("llama_32k", "minmax", units)


def test_group_selection_qwen_64k_per_kv_head_settings():
    # G = 7, block size and budget drawn per KV head (k equal within a group)
    units = [(0, 0), (5, 1), (9, 2), (15, 3)]
    _check_selection("qwen_64k", "minmax", units)


def test_group_decode_step_matches_oracle():
    wl, prob, dev, ws, summ, ks, nc, idx_ref, cnt_ref = _check_selection("tiny_4k", "minmax")
    idx = torch.full_like(idx_ref, -5)
    cnt = torch.full_like(cnt_ref, -5)
    out = torch.empty(wl.B, wl.Hq, wl.D, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    sa.decode_step(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ, idx, cnt,
                   out, lse, ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    assert torch.equal(cnt, cnt_ref)
    for b in range(wl.B):
        for h in range(wl.Hq):
            n = int(cnt[b, h])
            assert torch.equal(idx[b, h, :n], idx_ref[b, h, :n])
            # one list per group
            h0 = h - h % wl.G
            assert torch.equal(idx[b, h, :n], idx[b, h0, :n])
    sel = {(b, h): idx[b, h, :int(cnt[b, h])].cpu().numpy() for b in range(wl.B) for h in range(wl.Hq)}
    ref = H.oracle_decode(nc, wl, sel, sa.SEL_BLOCK, prob.scale)
    o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), (O, l) in ref.items():
        H.assert_close(o_np[b, h], O, f"group decode O (b={b}, h={h})")
        H.assert_close(np.array([l_np[b, h]]), np.array([l]), f"group decode lse (b={b}, h={h})")


def test_group_step_long_ragged_sequences_span_several_tile_windows():
    # more candidates than the fused select/build kernel holds: the group top-k
    # kernel, then one tile-builder CTA per 4096-page window; lengths end
    # inside window 2, on the window 0/1 edge, inside window 1 and at 0
    wl = synth.Workload("long_ragged", B=4, Hq=6, Hk=2, L=150000, lens=[150000, 65536, 70001, 0],
                        block_sizes=[16, 64], budget_bp=[500, 500], S=4, W=1024, c_heavy=2.0, heavy_count=6,
                        recency=2000)
    case = synth.make_decode_case(wl, 12)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks, selection=sa.SELECT_GROUP)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    idx = torch.full((wl.B, wl.Hq, prob.kcap), -5, dtype=torch.int32, device="cuda")
    cnt = torch.full((wl.B, wl.Hq), -5, dtype=torch.int32, device="cuda")
    out = torch.empty(wl.B, wl.Hq, wl.D, device="cuda")
    lse = torch.empty(wl.B, wl.Hq, device="cuda")
    sa.decode_step(prob, dev["q"], dev["k_pool"], dev["v_pool"], dev["page_table"], dev["seq_lens"], summ, idx, cnt,
                   out, lse, ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    ref = H.oracle_select_group(nc, wl, ks, "minmax")
    idx_np, cnt_np = idx.cpu().numpy(), cnt.cpu().numpy()
    for (b, h), (sel, _, _) in ref.items():
        assert np.array_equal(idx_np[b, h, :cnt_np[b, h]], sel), f"(b={b}, h={h}) group selection differs"
    dec = H.oracle_decode(nc, wl, {k: v[0] for k, v in ref.items()}, sa.SEL_BLOCK, prob.scale)
    o_np, l_np = out.cpu().numpy(), lse.cpu().numpy()
    for (b, h), (O, lz) in dec.items():
        H.assert_close(o_np[b, h], O, f"O(b={b},h={h})")
        H.assert_close(np.array([l_np[b, h]]), np.array([lz]), f"lse(b={b},h={h})")
