"""The benchmark's algorithmic-byte accounting (the numerator of its
roofline fraction) against an independent count from the oracle's token sets:
per (sequence, KV head) the K and V rows of the union over the group's heads
of I and J_h (read once per group), q, O + lse, and one page-table entry per
page read; the selection reads each candidate block's summary once per group.
CPU only."""
import numpy as np
import pytest
import torch

import bench
from oracle import sparse_attention_oracle as orc
from sparse_decode_attention_head_gb300 import sa, synth
from tests import harness as H


def _count(wl, nc, sel):
    D, G, P = wl.D, wl.G, wl.P
    dec = 0
    for b in range(wl.B):
        L = int(nc.seq_lens[b])
        for kvh in range(wl.Hk):
            Bs = wl.block_sizes[kvh]
            toks = set(orc.dense_tokens(L, wl.S, wl.W).tolist())
            for g in range(G):
                toks |= set(orc.sparse_tokens(L, wl.S, wl.W, Bs, sel[(b, kvh * G + g)][0]).tolist())
            pages = {t // P for t in toks}
            dec += len(toks) * (2 * D * 2) + G * D * 2 + G * (D * 4 + 4) + len(pages) * 4
    return dec


@pytest.mark.parametrize("name", ["tiny_4k", "ragged"])
def test_decode_bytes_match_an_independent_count(name):
    if name == "tiny_4k":
        wl = synth.workload("tiny_4k")
    else:   # block sizes 8 and 64 (half a page, four pages), ragged lengths
        wl = synth.Workload("ragged", B=3, Hq=6, Hk=2, L=1500, block_sizes=[8, 64], budget_bp=[1500, 800],
                            S=4, W=96, c_heavy=2.0, heavy_count=4, recency=300, lens=[1500, 1013, 333])
    case = synth.make_decode_case(wl, 2)
    nc = H.to_np_case(case)
    ks = synth.k_per_qhead(wl)
    prob = H.make_problem(wl, ks)
    sel = H.oracle_select(nc, wl, ks, "minmax")
    kcap = prob.kcap
    idx = torch.full((wl.B, wl.Hq, kcap), -1, dtype=torch.int32)
    cnt = torch.zeros(wl.B, wl.Hq, dtype=torch.int32)
    for (b, h), (s, _, _) in sel.items():
        idx[b, h, :len(s)] = torch.from_numpy(np.asarray(s, dtype=np.int32))
        cnt[b, h] = len(s)
    got = bench.algorithmic_bytes(wl, prob, nc.seq_lens, idx, cnt)
    assert got["decode"] == _count(wl, nc, sel)
    # selection: every candidate block's MINMAX summary (2 x D bf16) read once per group
    ncand = 0
    for b in range(wl.B):
        for kvh in range(wl.Hk):
            j0, j1 = orc.candidate_blocks(int(nc.seq_lens[b]), wl.S, wl.W, wl.block_sizes[kvh])
            ncand += j1 - j0
    assert got["select"] >= ncand * 2 * wl.D * 2
    assert got["total"] == got["decode"] + got["select"] + got["summary"]
