"""Appending the new token's K/V (sa_append_kv, sa_decode_step_append):
pool rows written bit for bit where the page table says, nothing else
touched, and the appending step equal to append + sa_decode_step."""
import pytest
import torch

from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _case(name, seed):
    wl = synth.workload(name)
    case = synth.make_decode_case(wl, seed)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    g = torch.Generator().manual_seed(seed + 1)
    k_new = torch.randn(wl.B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
    v_new = torch.randn(wl.B, wl.Hk, wl.D, generator=g).to(torch.bfloat16).cuda()
    return wl, prob, dev, k_new, v_new


def _write_rows(wl, dev, k_new, v_new, k_pool, v_pool):
    """The rows the append must write, done with tensor indexing."""
    pt = dev["page_table"].cpu()
    for b in range(wl.B):
        L = int(dev["seq_lens"][b])
        if L <= 0:
            continue
        phys = int(pt[b, (L - 1) // wl.P])
        k_pool[phys, :, (L - 1) % wl.P] = k_new[b]
        v_pool[phys, :, (L - 1) % wl.P] = v_new[b]


@pytest.mark.parametrize("name", ["tiny_4k", "llama_32k"])
def test_append_kv_writes_the_rows(name):
    wl, prob, dev, k_new, v_new = _case(name, 3)
    ws = sa.Workspace(prob)
    kp, vp = dev["k_pool"].clone(), dev["v_pool"].clone()
    sa.append_kv(prob, k_new, v_new, kp, vp, dev["page_table"], dev["seq_lens"], ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    kr, vr = dev["k_pool"].clone(), dev["v_pool"].clone()
    _write_rows(wl, dev, k_new, v_new, kr, vr)
    assert torch.equal(kp.view(torch.int16), kr.view(torch.int16))
    assert torch.equal(vp.view(torch.int16), vr.view(torch.int16))


@pytest.mark.parametrize("name", ["tiny_4k", "llama_32k"])
def test_decode_step_append_equals_append_then_step(name):
    wl, prob, dev, k_new, v_new = _case(name, 5)
    ws = sa.Workspace(prob)
    summ0 = H.gpu_summaries(prob, dev, ws)
    kcap = prob.kcap
    # reference: rows written by indexing, then the plain step
    kr, vr = dev["k_pool"].clone(), dev["v_pool"].clone()
    _write_rows(wl, dev, k_new, v_new, kr, vr)
    summ_r = summ0.clone()
    idx_r = torch.empty(wl.B, wl.Hq, kcap, dtype=torch.int32, device="cuda")
    cnt_r = torch.empty(wl.B, wl.Hq, dtype=torch.int32, device="cuda")
    o_r = torch.empty(wl.B, wl.Hq, wl.D, device="cuda")
    l_r = torch.empty(wl.B, wl.Hq, device="cuda")
    sa.decode_step(prob, dev["q"], kr, vr, dev["page_table"], dev["seq_lens"], summ_r, idx_r, cnt_r, o_r, l_r, ws)
    # the appending step on fresh copies of the pools and summaries
    kp, vp = dev["k_pool"].clone(), dev["v_pool"].clone()
    summ = summ0.clone()
    idx = torch.full_like(idx_r, -5)
    cnt = torch.full_like(cnt_r, -5)
    out = torch.full_like(o_r, float("nan"))
    lse = torch.full_like(l_r, float("nan"))
    sa.decode_step_append(prob, dev["q"], k_new, v_new, kp, vp, dev["page_table"], dev["seq_lens"], summ, idx, cnt,
                          out, lse, ws)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    assert torch.equal(kp.view(torch.int16), kr.view(torch.int16))
    assert torch.equal(vp.view(torch.int16), vr.view(torch.int16))
    assert torch.equal(summ.view(torch.int16), summ_r.view(torch.int16))   # tail summary from the new row
    assert torch.equal(cnt, cnt_r)
    for b in range(wl.B):
        for h in range(wl.Hq):
            n = int(cnt[b, h])
            assert torch.equal(idx[b, h, :n], idx_r[b, h, :n])
    H.assert_close(out.cpu().numpy(), o_r.cpu().numpy(), "append step O")
    H.assert_close(lse.cpu().numpy(), l_r.cpu().numpy(), "append step lse")
    # and the new row is really used: the summary of the tail block changed
    L = int(dev["seq_lens"][0])
    j = (L - 1) // wl.block_sizes[0]
    assert not torch.equal(summ[0, 0, j].view(torch.int16), summ0[0, 0, j].view(torch.int16))
