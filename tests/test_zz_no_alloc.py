"""sa_sparse_decode_noalloc: the decode step for callers that cannot allocate
device memory (for example inside a framework that owns every allocation
through its own pool), so cannot pass sa_sparse_decode a workspace.

Called through the C ABI; its output must match sa_sparse_decode's within the
tolerance the parity tests use, on two calls in a row (the second call finds
the library's fixed scratch holding the first call's contents).  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H

pytestmark = pytest.mark.gpu


def _noalloc(prob, dev, idx, cnt, gran, status):
    out = torch.full((prob.B, prob.Hq, prob.D), float("nan"), device="cuda")
    lse = torch.full((prob.B, prob.Hq), float("nan"), device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = sa.lib().sa_sparse_decode_noalloc(
        prob.ref, p(dev["q"]), p(dev["k_pool"]), p(dev["v_pool"]), p(dev["page_table"]), p(dev["seq_lens"]),
        p(idx), p(cnt), gran, p(out), p(lse), None, None if status is None else p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == sa.SA_OK, sa.status_string(rc)
    return out, lse


@pytest.mark.parametrize("name", ["tiny_4k", "ragged"])
def test_noalloc_matches_workspace_decode_twice(name):
    if name == "tiny_4k":
        wl = synth.workload("tiny_4k")
    else:
        wl = synth.Workload("ragged", B=3, Hq=6, Hk=2, L=1500, block_sizes=[8, 64], budget_bp=[1500, 800],
                            S=4, W=96, c_heavy=2.0, heavy_count=4, recency=300, lens=[1500, 1013, 333])
    case = synth.make_decode_case(wl, 21)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    idx, cnt, _ = H.gpu_select(prob, dev, summ, ws, with_scores=False)
    ref_o, ref_l = H.gpu_decode(prob, dev, idx, cnt, ws)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        o, l = _noalloc(prob, dev, idx, cnt, sa.SEL_BLOCK, status)
        torch.cuda.synchronize()
        H.assert_close(o.cpu().numpy(), ref_o.cpu().numpy(), "noalloc O")
        H.assert_close(l.cpu().numpy(), ref_l.cpu().numpy(), "noalloc lse")
        assert int(status.item()) == sa.SA_OK


def test_noalloc_vs_oracle_long_ragged_given_oracle_selections():
    # the oracle's own index sets in, the fp64 oracle's O and lse out:
    # lengths past 4096 pages (tile-list windows), ending inside window 2, on
    # the window 0/1 edge, inside window 1, and at 0 (O = 0, lse = -inf)
    wl = synth.Workload("long_ragged", B=4, Hq=6, Hk=2, L=150000, lens=[150000, 65536, 70001, 0],
                        block_sizes=[16, 64], budget_bp=[500, 500], S=4, W=1024, c_heavy=2.0, heavy_count=6,
                        recency=2000)
    case = synth.make_decode_case(wl, 23)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    ref_sel = H.oracle_select(nc, wl, ks, "minmax")
    idx, cnt = H.sel_to_tensor(prob, {k: v[0] for k, v in ref_sel.items()})
    dev = H.to_dev(case)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    o, l = _noalloc(prob, dev, idx, cnt, sa.SEL_BLOCK, status)
    torch.cuda.synchronize()
    assert int(status.item()) == sa.SA_OK
    ref = H.oracle_decode(nc, wl, {k: v[0] for k, v in ref_sel.items()}, sa.SEL_BLOCK, prob.scale)
    on, ln = o.cpu().numpy(), l.cpu().numpy()
    for (b, h), (O, lz) in ref.items():
        H.assert_close(on[b, h], O, f"noalloc O(b={b},h={h})")
        H.assert_close(np.array([ln[b, h]]), np.array([lz]), f"noalloc lse(b={b},h={h})")


def _tiny_setup(seed):
    wl = synth.workload("tiny_4k")
    case = synth.make_decode_case(wl, seed)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    dev = H.to_dev(case)
    ws = sa.Workspace(prob)
    summ = H.gpu_summaries(prob, dev, ws)
    idx, cnt, _ = H.gpu_select(prob, dev, summ, ws, with_scores=False)
    ref_o, ref_l = H.gpu_decode(prob, dev, idx, cnt, ws)
    return prob, dev, idx, cnt, ref_o, ref_l


def test_noalloc_without_a_status_word():
    # status_or_null = NULL: the status lives in the library's scratch; the
    # outputs are what counts
    prob, dev, idx, cnt, ref_o, ref_l = _tiny_setup(22)
    for _ in range(2):
        o, l = _noalloc(prob, dev, idx, cnt, sa.SEL_BLOCK, None)
        torch.cuda.synchronize()
        H.assert_close(o.cpu().numpy(), ref_o.cpu().numpy(), "noalloc O (no status word)")
        H.assert_close(l.cpu().numpy(), ref_l.cpu().numpy(), "noalloc lse (no status word)")


def test_noalloc_clears_a_stale_status():
    # a status word left holding an error code from earlier reads SA_OK after a clean call
    prob, dev, idx, cnt, ref_o, ref_l = _tiny_setup(23)
    status = torch.full((1,), sa.SA_ERR_TIMEOUT, dtype=torch.int32, device="cuda")
    o, l = _noalloc(prob, dev, idx, cnt, sa.SEL_BLOCK, status)
    torch.cuda.synchronize()
    assert int(status.item()) == sa.SA_OK
    H.assert_close(o.cpu().numpy(), ref_o.cpu().numpy(), "noalloc O")


def test_noalloc_rejects_problem_larger_than_its_scratch():
    wl = synth.workload("llama_32k")
    prob = sa.Problem(B=64, Hq=32, Hk=8, max_pages_per_seq=16384, num_pages=1 << 16, sink=4, window=1024,
                      block_sizes=[16] * 8, k_per_head=[100] * 32, kcap=100)
    v = ctypes.c_void_p(256)   # never dereferenced: the size check fails first
    rc = sa.lib().sa_sparse_decode_noalloc(prob.ref, v, v, v, v, v, v, v, 0, v, v, None, None, None)
    assert rc == sa.SA_ERR_CAPACITY
