"""Benchmark: one decode step of hybrid sparse attention on the Llama-3.1-8B
shaped 32K layer (B=8, 32 query / 8 KV heads, D=128, page = block = 16,
5 % budget, 4 sinks, 1024-token window), bf16 paged KV.

A step is the whole hot path for one layer:
  tail-block summary refresh -> fused block score + per-head top-k ->
  paged sparse decode (dense sinks + window, sparse selected blocks, exact
  log-sum-exp merge of the split-K partials).
Eight independent layer copies (8.6 GB of KV) rotate from step to step, so
nothing a step reads is still in the 129 MB L2 when it is read again.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_decode_attention_head_gb300 import sa, synth  # noqa: E402

WORKLOAD = "llama_32k"
N_LAYERS = 8   # default; --layers overrides
METRIC = "decode attn queries/s & achieved HBM GB/s (% of 8 TB/s), Llama-3-8B shape 32K"
FALLBACK_HBM_GBS = 6800.0
PROFILE = os.path.join(ROOT, "profiles", "sparse_decode_llama_32k.md")


# --------------------------------------------------------------------------- helpers

def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# kernels of one sa_decode_step on this workload: scores, fused top-k + tile build + tail summary,
# decode, chunk merge
STEP_LAUNCHES = 4


def reduce_max_ms(ms, world, device):
    """Maximum over the ranks of a per-rank duration; every rank gets it."""
    if world == 1:
        return float(ms)
    import torch.distributed as dist
    t = torch.tensor([float(ms)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(world, queries_per_step, steps, max_ms):
    """Queries per second of the whole job: every rank decodes its own batch
    each step (replicas), timed by the slowest rank."""
    return world * queries_per_step * steps / (max_ms / 1e3)


def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "sa_common.cuh"):
        with open(os.path.join(ROOT, "sparse_decode_attention_head_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """dram bytes per launch of the decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    try:
        txt = open(PROFILE).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", txt)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m_hash or not m_tr or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_tr.group(1))


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- our arm

def unit_decode_bytes(L, S, W, Bs, P, D, G, sel_lists):
    """Algorithmic bytes of the decode for one (sequence, KV head): the K and
    V rows of I U (union over the group's heads of their selected blocks
    inside M), read once per group, q, O + lse, one page-table entry per page."""
    s_end = min(S, L)
    w_beg = max(L - W, s_end)
    att = np.zeros(max(L, 1), dtype=bool)
    att[:s_end] = True
    att[w_beg:L] = True
    for ids in sel_lists:
        ids = np.asarray(ids, dtype=np.int64)
        if ids.size == 0:
            continue
        t = (ids[:, None] * Bs + np.arange(Bs)[None, :]).ravel()
        t = t[(t >= s_end) & (t < w_beg)]
        att[t] = True
    att = att[:L]
    ntok = int(att.sum())
    npages = int(np.unique(np.nonzero(att)[0] // P).size)
    return ntok * 2 * D * 2 + G * D * 2 + G * (D * 4 + 4) + npages * 4


def algorithmic_bytes(wl, prob, seq_lens, sel_idx, sel_cnt):
    """Per-step algorithmic HBM bytes, split by call (byte accounting of the
    hot-path scope: summaries of candidate blocks, KV rows of I U (union of the
    group's selected blocks) once per group, q, O + lse, page-table entries)."""
    P, D, G = wl.P, wl.D, wl.G
    si = sel_idx.cpu().numpy() if hasattr(sel_idx, "cpu") else np.asarray(sel_idx)
    sc = sel_cnt.cpu().numpy() if hasattr(sel_cnt, "cpu") else np.asarray(sel_cnt)
    dec = sel = summ = 0
    summ_row = 2 * D * 2 if prob.mode == sa.SUMMARY_MINMAX else D * 2
    for b in range(wl.B):
        L = int(seq_lens[b])
        for kvh in range(wl.Hk):
            Bs = wl.block_sizes[kvh]
            j0, j1 = synth.candidate_range(L, wl.S, wl.W, Bs)
            lists = [si[b, kvh * G + g, :sc[b, kvh * G + g]] for g in range(G)]
            dec += unit_decode_bytes(L, wl.S, wl.W, Bs, P, D, G, lists)
            sel += (j1 - j0) * summ_row + G * D * 2 + G * 4 * (1 + int(np.mean(sc[b, kvh * G:(kvh + 1) * G])))
            summ += Bs * D * 2 + summ_row + ((Bs + P - 1) // P) * 4
    return {"decode": dec, "select": sel, "summary": summ, "total": dec + sel + summ}


def run_ours(args):
    world, rank, local = dist_info()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    sa.lib()

    wl = synth.workload(WORKLOAD)
    ks = synth.k_per_qhead(wl)
    kcap = max(ks)
    prob = sa.Problem(B=wl.B, Hq=wl.Hq, Hk=wl.Hk, max_pages_per_seq=wl.max_pages_per_seq,
                      num_pages=wl.B * wl.max_pages_per_seq, sink=wl.S, window=wl.W,
                      block_sizes=wl.block_sizes, k_per_head=ks, kcap=kcap, mode=sa.SUMMARY_MINMAX)
    ws = sa.Workspace(prob, device=dev)

    global N_LAYERS
    N_LAYERS = args.layers
    layers = []
    for l in range(N_LAYERS):
        c = synth.make_decode_case(wl, 1000 * rank + 100 + l, device=dev)
        summ = torch.empty(prob.summary_shape(), dtype=torch.bfloat16, device=dev)
        sa.block_summarize(prob, c.k_pool, c.page_table, c.seq_lens, summ, ws)   # one-time full build
        layers.append(dict(q=c.q, k=c.k_pool, v=c.v_pool, pt=c.page_table, sl=c.seq_lens, summ=summ,
                           sel_idx=torch.empty(wl.B, wl.Hq, kcap, dtype=torch.int32, device=dev),
                           sel_cnt=torch.empty(wl.B, wl.Hq, dtype=torch.int32, device=dev)))
        del c
    torch.cuda.synchronize()
    out = torch.empty(wl.B, wl.Hq, wl.D, dtype=torch.float32, device=dev)
    lse = torch.empty(wl.B, wl.Hq, dtype=torch.float32, device=dev)

    def sub_select(L):
        sa.block_summarize(prob, L["k"], L["pt"], L["sl"], L["summ"], ws, block_begin=sa.BLOCKS_TAIL)
        sa.select_topk(prob, L["q"], L["summ"], L["sl"], L["sel_idx"], L["sel_cnt"], ws)

    def sub_decode(L):
        sa.sparse_decode(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["sel_idx"], L["sel_cnt"], out, lse, ws)

    def whole_step(L):   # the hot path in one call: tail summary, scores, top-k, decode
        sa.decode_step(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["sel_idx"], L["sel_cnt"], out,
                       lse, ws)

    # eager warm-up (sets kernel attributes, selection for the byte count)
    for L in layers:
        sub_select(L)
        sub_decode(L)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    nbytes = [algorithmic_bytes(wl, prob, L["sl"].cpu().numpy(), L["sel_idx"], L["sel_cnt"]) for L in layers]

    # The timed work is captured once into CUDA graphs holding all K steps, so
    # the GPU runs them back to back whatever the host's launch rate:
    #   g_step: K whole steps (sa_decode_step), layers rotating;
    #   g_dec / g_sel: the K decode calls / the K select calls alone, for the
    #   per-kernel averages the roofline uses.
    K, W = args.steps, args.warmup
    stream = torch.cuda.Stream(device=dev)

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(K):
                    fn(layers[(W + i) % N_LAYERS])
        return g

    g_step = capture(whole_step)
    g_dec = capture(sub_decode)
    g_sel = capture(sub_select)
    torch.cuda.synchronize()

    # the group-shared selection variant (one top-k per KV head for its query
    # heads): same layers, its own selection buffers, timed the same way
    prob_g = None
    if not args.no_group:
        prob_g = sa.Problem(B=wl.B, Hq=wl.Hq, Hk=wl.Hk, max_pages_per_seq=wl.max_pages_per_seq,
                            num_pages=wl.B * wl.max_pages_per_seq, sink=wl.S, window=wl.W,
                            block_sizes=wl.block_sizes, k_per_head=ks, kcap=kcap, mode=sa.SUMMARY_MINMAX,
                            selection=sa.SELECT_GROUP)
        ws_g = sa.Workspace(prob_g, device=dev)
        for L in layers:
            L["sel_idx_g"] = torch.empty_like(L["sel_idx"])
            L["sel_cnt_g"] = torch.empty_like(L["sel_cnt"])

        def group_step(L):
            sa.decode_step(prob_g, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["sel_idx_g"],
                           L["sel_cnt_g"], out, lse, ws_g)

        for L in layers:
            group_step(L)
        torch.cuda.synchronize()
        assert ws_g.status() == sa.SA_OK
        nbytes_g = [algorithmic_bytes(wl, prob_g, L["sl"].cpu().numpy(), L["sel_idx_g"], L["sel_cnt_g"])
                    for L in layers]
        g_group = capture(group_step)
        torch.cuda.synchronize()

    R = args.repeats

    with torch.cuda.stream(stream):   # warm-up steps, eager
        for i in range(W):
            sub_select(layers[i % N_LAYERS])
            sub_decode(layers[i % N_LAYERS])
    for g in (g_dec, g_sel, g_step):  # first replays upload the graphs
        replay_ms(g, stream, 1)
    if prob_g is not None:
        replay_ms(g_group, stream, 1)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    torch.cuda.synchronize()
    # each graph replayed R times, every replay its own K-step timed window
    step_reps = replay_ms(g_step, stream, R)
    dec_reps = replay_ms(g_dec, stream, R)
    sel_reps = replay_ms(g_sel, stream, R)
    group = None
    if prob_g is not None:
        g_sp = spread(replay_ms(g_group, stream, R), K)
        g_ms = g_sp["median_ms_per_step"]
        g_bytes = float(np.mean([nbytes_g[(W + i) % N_LAYERS]["total"] for i in range(K)]))
        group = {"selection": "one top-k per KV head over the fp32 sum of its query heads' scores (a variant; "
                              "the headline selects per head)",
                 "ms_per_step": g_ms, "spread": g_sp, "value": round(wl.B * wl.Hq / (g_ms / 1e3), 1),
                 "unit": "queries/s", "algorithmic_bytes_per_step": int(g_bytes),
                 "achieved_gbs": round(g_bytes / (g_ms / 1e3) / 1e9, 1)}
    clk = clocks.stop()
    step_sp, dec_sp, sel_sp = spread(step_reps, K), spread(dec_reps, K), spread(sel_reps, K)
    total_ms = reduce_max_ms(float(np.median(step_reps)), world, dev)   # median K-step window, slowest rank
    ms_step = total_ms / K
    queries = wl.B * wl.Hq
    value = whole_job_value(world, queries, K, total_ms)

    layer_of = [(W + i) % N_LAYERS for i in range(K)]
    dec_bytes = float(np.mean([nbytes[l]["decode"] for l in layer_of]))
    step_bytes = float(np.mean([nbytes[l]["total"] for l in layer_of]))
    dec_avg_ms = dec_sp["median_ms_per_step"]
    peak, peak_src = measured_hbm_peak()
    achieved = dec_bytes / (dec_avg_ms / 1e3) / 1e9

    # end to end through the public binding: pinned host q in, O + lse out
    e2e = None
    if not args.no_e2e:
        # the prepared plan (one graph launch a step) is the headline: the eager
        # path spends longer enqueueing a step on the host than the GPU spends
        # running it; eager launches are reported beside it
        e2e = run_e2e(args, prob, layers, ws, out, lse, dev, prepared=True)
        e2e["eager_launches"] = {k: v for k, v in run_e2e(args, prob, layers, ws, out, lse, dev, prepared=False).items()
                                 if k in ("value", "ms_per_step", "host_enqueue_ms_per_step", "serial_ms_per_step",
                                          "path")}
    tables = None if args.no_tables else run_tables(args, dev)
    bypass = None if args.no_bypass else run_bypass(args, dev, rank)
    config2 = None if args.no_config2 else run_qwen(args, dev, rank)
    gpu_launches = STEP_LAUNCHES * K

    res = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "queries/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V with planted sink, heavy blocks and recency ramp)",
        "config": headline_config(world),
        "timing": {"method": f"CUDA events around each of {R} replays of one CUDA graph of K = {K} steps; "
                             "value and ms_per_step from the median replay",
                   "l2": f"{N_LAYERS} rotating independent layer copies ({N_LAYERS * 1.07:.1f} GB KV), inputs > L2",
                   "repeats": R},
        "spread": step_sp,
        "roofline": {"bound": "hbm", "kernel": "sa_sparse_decode (tile build + paged decode + split-K merge), timed alone",
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(),
                     "algorithmic_bytes_per_launch": int(dec_bytes), "avg_launch_ms": round(dec_avg_ms, 5),
                     "spread": dec_sp},
        "step_roofline": {"achieved_gbs": round(step_bytes / (ms_step / 1e3) / 1e9, 1),
                          "frac": round(step_bytes / (ms_step / 1e3) / 1e9 / peak, 4),
                          "algorithmic_bytes_per_step": int(step_bytes),
                          "select_avg_ms": sel_sp["median_ms_per_step"], "select_spread": sel_sp},
        "e2e": e2e,
        "tables_roofline": tables,
        "config2": config2,
        "group_select_variant": group,
        "bypass_variant": bypass,
        "gpu_launches": gpu_launches,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline_cells(args, dev, layers[0], wl, ks, prob.scale)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)


def headline_config(world):
    """The workload the headline is quoted on (both arms print this)."""
    wl = synth.workload(WORKLOAD)
    return {"workload": "llama3.1-8b layer, decode, B8 x 32q/8kv heads x D128, ctx 32768, "
                        "page=block=16, budget 5% (k=100 blocks), sinks 4, window 1024, minmax summaries",
            "global_batch": wl.B, "seq_len": wl.L, "parallelism": f"replicas x{world}"}


def replay_ms(g, stream, reps):
    """Milliseconds of each of `reps` replays of graph g, CUDA events on the
    launching stream, the device synchronised on both sides of every replay."""
    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1))
    return out


def spread(reps_ms, steps):
    """Median, p10 and p90 of the per-step time over the replays."""
    a = np.asarray(reps_ms, dtype=np.float64) / steps
    return {"median_ms_per_step": round(float(np.median(a)), 5), "p10_ms_per_step": round(float(np.percentile(a, 10)), 5),
            "p90_ms_per_step": round(float(np.percentile(a, 90)), 5), "repeats": int(a.size)}


def run_e2e(args, prob, layers, ws, out, lse, dev, prepared=True):
    """End to end through the public binding: every step copies its q in from
    pinned host memory and its (O, lse) back out.  Measured twice: copies and
    the step serialised on one stream, and pipelined (the next step's q copied
    in on an input stream and the previous step's result read back on an
    output stream while the current step computes, result buffers
    double-buffered); every copy of the K steps completes inside the timed
    region in both."""
    wl_B, Hq, D = prob.B, prob.Hq, prob.D
    q_host = [L["q"].cpu().pin_memory() for L in layers]
    nres = wl_B * Hq * (D + 1)
    # O and lse share one device buffer, so a step's result comes back in one copy
    res = [torch.empty(nres, dtype=torch.float32, device=dev) for _ in range(2)]
    res_host = [torch.empty(nres, dtype=torch.float32).pin_memory() for _ in range(2)]
    views = [(r[:wl_B * Hq * D].view(wl_B, Hq, D), r[wl_B * Hq * D:].view(wl_B, Hq)) for r in res]
    K, W = args.steps, args.warmup

    # prepared: sa.StepPlan (the step captured once per buffer set inside the
    # library, one graph launch a step); else sa.DecodeStepCall (marshalled
    # once, the step's kernels launched eagerly each step)
    make = sa.StepPlan if prepared else sa.DecodeStepCall
    calls = [[make(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["sel_idx"], L["sel_cnt"], o, l, ws)
              for (o, l) in views] for L in layers]

    def decode(i, r):
        calls[i % N_LAYERS][r]()

    def serial_step(i):
        layers[i % N_LAYERS]["q"].copy_(q_host[i % N_LAYERS], non_blocking=True)
        decode(i, 0)
        res_host[0].copy_(res[0], non_blocking=True)

    main = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    q_ready = [torch.cuda.Event() for _ in range(N_LAYERS)]
    q_free = [torch.cuda.Event() for _ in range(N_LAYERS)]
    done = [torch.cuda.Event() for _ in range(2)]
    read = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        j = i % N_LAYERS
        with torch.cuda.stream(s_in):
            s_in.wait_event(q_free[j])          # the step that last read this q has finished
            layers[j]["q"].copy_(q_host[j], non_blocking=True)
            q_ready[j].record(s_in)

    def pipelined(first, n):
        for e in q_free:
            e.record(main)
        for e in read:
            e.record(main)
        copy_in(first)
        for i in range(first, first + n):
            if i + 1 < first + n:
                copy_in(i + 1)
            j, r = i % N_LAYERS, i % 2
            main.wait_event(q_ready[j])
            main.wait_event(read[r])              # the result buffer has been read back
            decode(i, r)
            q_free[j].record(main)
            done[r].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done[r])
                res_host[r].copy_(res[r], non_blocking=True)
                read[r].record(s_out)
        main.wait_stream(s_out)

    def timed(fn):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(main)
        t0 = time.perf_counter()
        fn()
        host_s = time.perf_counter() - t0
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1), host_s

    for i in range(W):
        serial_step(i)
    ms_serial, _ = timed(lambda: [serial_step(W + i) for i in range(K)])
    pipelined(0, W)
    ms, host_s = timed(lambda: pipelined(W, K))
    return {"value": round(wl_B * Hq * K / (ms / 1e3), 1), "unit": "queries/s",
            "h2d_bytes_per_step": wl_B * Hq * D * 2, "d2h_bytes_per_step": nres * 4,
            "ms_per_step": round(ms / K, 5), "host_enqueue_ms_per_step": round(host_s * 1e3 / K, 5),
            "serial_ms_per_step": round(ms_serial / K, 5),
            "path": ("python binding (sa.StepPlan) -> sa_step_plan_launch (C-ABI): the step captured once per buffer "
                     "set inside the library, one graph launch a step" if prepared else
                     "python binding (sa.DecodeStepCall) -> sa_decode_step (C-ABI), eager launches") +
                    "; q in and (O, lse) out copied on their own streams, overlapping the neighbouring steps"}


def run_tables(args, dev, reps=100):
    """Step a7 on the 128K table workload (B4, 32q/8kv, L 131072 + 1 per step):
    sa_update_score_tables alone, in a CUDA graph of `reps` launches that
    alternate the two table buffers, fed by one real decode step (its
    selections, logits and lse).  The 4 x 64 MB tables and their 256 MB of
    reads + writes per launch are larger than L2."""
    wl = synth.table_workload("tables_128k")
    case = synth.make_table_case(wl, 7, device=dev)
    B, Hq, Hk = wl.B, wl.Hq, wl.Hk
    mpp = wl.max_pages_per_seq
    N = mpp * wl.P
    prob = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                      block_sizes=[16] * Hk, k_per_head=[0] * Hq, kcap=wl.kcap)
    ws = sa.Workspace(prob, device=dev)
    tv = [case.vert0, torch.empty(B, Hq, N, device=dev)]
    ts = [case.slash0, torch.empty(B, Hq, N, device=dev)]
    cand = [torch.zeros(B, Hq, wl.kcap, dtype=torch.int32, device=dev) for _ in range(2)]
    cnt = [torch.zeros(B, Hq, dtype=torch.int32, device=dev) for _ in range(2)]
    logits = torch.zeros(B, Hq, N, device=dev)
    out = torch.empty(B, Hq, wl.D, device=dev)
    lse = torch.empty(B, Hq, device=dev)
    L0 = wl.L0
    sl0 = torch.full((B,), L0, dtype=torch.int32, device=dev)
    sl1 = torch.full((B,), L0 + 1, dtype=torch.int32, device=dev)
    # one real step: first update (tables carried over), decode over I + candidates with logits
    sa.update_score_tables(prob, tv[0], ts[0], tv[1], ts[1], sl0, cand[0], cnt[0], ws, beta=wl.beta)
    sa.sparse_decode(prob, case.q_steps[0], case.k_pool, case.v_pool, case.page_table, sl0, cand[0], cnt[0], out,
                     lse, ws, granularity=sa.SEL_TOKEN, logits=logits)
    prev = dict(prev_seq_lens=sl0, prev_sel_idx=cand[0], prev_sel_cnt=cnt[0], prev_logits=logits, prev_lse=lse)
    torch.cuda.synchronize()
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()

    def update(i):
        a, b = i % 2, (i + 1) % 2
        sa.update_score_tables(prob, tv[b], ts[b], tv[a], ts[a], sl1, cand[1], cnt[1], ws, beta=wl.beta, prev=prev)

    with torch.cuda.stream(st):
        for i in range(3):
            update(i)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st, capture_error_mode="relaxed"):
            for i in range(reps):
                update(i)
    replay_ms(g, st, 1)
    tab_sp = spread(replay_ms(g, st, args.repeats), reps)
    ms = tab_sp["median_ms_per_step"]
    status = ws.status()
    # algorithmic bytes: both tables read and written, the previous step's logits at
    # its attended positions, its selection list, and the new candidate list
    n_att = wl.S + wl.W + cnt[0].sum().item() / (B * Hq)
    per_head = 4 * N * 4 + n_att * 4 + cnt[0].float().mean().item() * 4 + cnt[1].float().mean().item() * 4
    nbytes = B * Hq * per_head
    peak, peak_src = measured_hbm_peak()
    achieved = nbytes / (ms / 1e3) / 1e9
    # exact top-k inside the candidates (16 tokens a head), timed the same way
    prob_t = sa.Problem(B=B, Hq=Hq, Hk=Hk, max_pages_per_seq=mpp, num_pages=B * mpp, sink=wl.S, window=wl.W,
                        block_sizes=[16] * Hk, k_per_head=[16] * Hq, kcap=wl.kcap)
    tsel = torch.empty(B, Hq, wl.kcap, dtype=torch.int32, device=dev)
    tcnt = torch.empty(B, Hq, dtype=torch.int32, device=dev)
    q1 = case.q_steps[1]
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        for i in range(3):
            sa.select_tokens(prob_t, q1, case.k_pool, case.page_table, sl1, cand[1], cnt[1], tsel, tcnt, ws)
        torch.cuda.synchronize()
        with torch.cuda.graph(g2, stream=st, capture_error_mode="relaxed"):
            for i in range(reps):
                sa.select_tokens(prob_t, q1, case.k_pool, case.page_table, sl1, cand[1], cnt[1], tsel, tcnt, ws)
    replay_ms(g2, st, 1)
    ms_tok = spread(replay_ms(g2, st, args.repeats), reps)["median_ms_per_step"]
    n_cand = cnt[1].sum().item()
    tok_bytes = n_cand * (wl.D * 2 + 4 + 4 + 4) + B * Hq * (wl.D * 2 + 16 * 4 + 8)
    token_topk = {"kernel": "sa_select_tokens (canonical q.k over each head's candidates, top 16)",
                  "avg_launch_ms": round(ms_tok, 5), "candidates": int(n_cand),
                  "algorithmic_bytes_per_launch": int(tok_bytes),
                  "achieved_gbs": round(tok_bytes / (ms_tok / 1e3) / 1e9, 1),
                  "note": "a few KB a head: launch and latency bound, not bandwidth bound"}
    return {"workload": "score tables, B4 x 32q/8kv heads, L 131072 + 1, tables fp32 [4][32][131136] x2",
            "kernel": "sa_update_score_tables (decay, threshold, expansion in one pass)",
            "avg_launch_ms": round(ms, 5), "spread": tab_sp, "algorithmic_bytes_per_launch": int(nbytes),
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "mean_candidates_per_head": round(cnt[1].float().mean().item(), 1), "status": status,
            "exact_token_topk": token_topk}


def run_bypass(args, dev, rank, reps=200):
    """The head-sparsity bypass (LFPS Algorithm 1 step 1, epsilon 0.85) on the
    32K Llama shape with 4 of 32 query heads per sequence aligned with key 0
    and no sink planted in the keys (llama_32k_sinkheads): sa_decode_step
    against sa_decode_step_bypass on the same rotating layer copies, each a
    CUDA graph of `reps` steps."""
    wl = synth.workload("llama_32k_sinkheads")
    ks = synth.k_per_qhead(wl)
    kcap = max(ks)
    prob = sa.Problem(B=wl.B, Hq=wl.Hq, Hk=wl.Hk, max_pages_per_seq=wl.max_pages_per_seq,
                      num_pages=wl.B * wl.max_pages_per_seq, sink=wl.S, window=wl.W,
                      block_sizes=wl.block_sizes, k_per_head=ks, kcap=kcap, mode=sa.SUMMARY_MINMAX)
    ws = sa.Workspace(prob, device=dev)
    layers = []
    for l in range(N_LAYERS):
        c = synth.make_decode_case(wl, 1000 * rank + 500 + l, device=dev)
        summ = torch.empty(prob.summary_shape(), dtype=torch.bfloat16, device=dev)
        sa.block_summarize(prob, c.k_pool, c.page_table, c.seq_lens, summ, ws)
        st = torch.empty(sa.kv_stats_shape(prob), device=dev)
        sa.kv_stats(prob, c.k_pool, c.v_pool, c.page_table, c.seq_lens, st, ws)
        layers.append(dict(q=c.q, k=c.k_pool, v=c.v_pool, pt=c.page_table, sl=c.seq_lens, summ=summ, st=st,
                           sel_idx=torch.empty(wl.B, wl.Hq, kcap, dtype=torch.int32, device=dev),
                           sel_cnt=torch.empty(wl.B, wl.Hq, dtype=torch.int32, device=dev),
                           byp=torch.empty(wl.B, wl.Hq, dtype=torch.int32, device=dev)))
        del c
    out = torch.empty(wl.B, wl.Hq, wl.D, device=dev)
    lse = torch.empty(wl.B, wl.Hq, device=dev)

    def plain(L):
        sa.decode_step(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["sel_idx"], L["sel_cnt"], out,
                       lse, ws)

    def bypass(L):
        sa.decode_step_bypass(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["st"], L["sel_idx"],
                              L["sel_cnt"], out, lse, L["byp"], ws)

    stream = torch.cuda.Stream(device=dev)
    res = {}
    for name, fn in (("plain", plain), ("bypass", bypass)):
        with torch.cuda.stream(stream):
            for L in layers:
                fn(L)
        torch.cuda.synchronize()
        if name == "bypass":
            frac = float(np.mean([L["byp"].float().mean().item() for L in layers]))
            nbytes = []
            for L in layers:
                nb = algorithmic_bytes(wl, prob, L["sl"].cpu().numpy(), L["sel_idx"], L["sel_cnt"])["total"]
                # the estimate: sink + 6 window key rows and the sums per KV head, q per head,
                # the mean row and lse per bypassed head
                nb += wl.B * wl.Hk * (7 * wl.D * 2 + 3 * wl.D * 4) + wl.B * wl.Hq * (wl.D * 2 + 8)
                nb += int(L["byp"].sum().item()) * (wl.D * 4 + 4)
                nbytes.append(nb)
        else:
            nbytes = [algorithmic_bytes(wl, prob, L["sl"].cpu().numpy(), L["sel_idx"], L["sel_cnt"])["total"]
                      for L in layers]
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for i in range(reps):
                    fn(layers[i % N_LAYERS])
        replay_ms(g, stream, 1)
        sp = spread(replay_ms(g, stream, max(5, args.repeats // 3)), reps)
        ms = sp["median_ms_per_step"]
        b = float(np.mean([nbytes[i % N_LAYERS] for i in range(reps)]))
        res[name] = {"ms_per_step": round(ms, 5), "spread": sp, "value": round(wl.B * wl.Hq / (ms / 1e3), 1),
                     "unit": "queries/s", "algorithmic_bytes_per_step": int(b),
                     "achieved_gbs": round(b / (ms / 1e3) / 1e9, 1)}
        del g
    assert ws.status() == sa.SA_OK
    return {"workload": "llama3.1-8b layer shape, ctx 32768, B8, 4 of 32 query heads per sequence "
                        "sink-dominated (q aligned with key 0), no key sink; epsilon 0.85",
            "bypassed_head_fraction": round(frac, 4),
            "step_plain": res["plain"], "step_bypass": res["bypass"],
            "speedup": round(res["plain"]["ms_per_step"] / res["bypass"]["ms_per_step"], 3)}


SWEEP_BATCH = (1, 4, 16, 64)
SWEEP_CTX = (8192, 32768, 131072, 262144)
SWEEP_BUDGET_BP = (100, 500, 1000, 10000)
SWEEP_LAYERS = 32
SWEEP_STEPS = 16
SWEEP_KV_CAP = 150e9


def run_sweep(args):
    """The throughput sweep of the full decode-attention stack: 32
    Llama-3-8B-shaped layers (distinct KV caches), batch x context x budget,
    16 decode steps each appending one token per sequence per layer
    (sa_decode_step_append), cells whose KV exceeds 150 GB left out.  The
    16 x 32 layer-steps of a cell are one CUDA graph, replayed between CUDA
    events.  One JSON line per cell."""
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sa.lib()
    st = torch.cuda.Stream(device=dev)
    only = None   # --sweep-cells B:ctx:bp,... restricts the sweep to those cells
    if args.sweep_cells:
        only = {tuple(int(v) for v in c.split(":")) for c in args.sweep_cells.split(",")}
    for B in SWEEP_BATCH:
        for ctx in SWEEP_CTX:
            budgets = [bp for bp in SWEEP_BUDGET_BP if only is None or (B, ctx, bp) in only]
            if not budgets:
                continue
            kv = SWEEP_LAYERS * B * ctx * 8 * 16 * 128 * 2 * 2 / 16
            if kv > SWEEP_KV_CAP:
                print(json.dumps({"sweep_cell": {"batch": B, "context": ctx}, "skipped": f"KV {kv / 1e9:.0f} GB > 150 GB"}),
                      flush=True)
                continue
            base = synth.sweep_workload(B, ctx, budgets[0], extra_tokens=SWEEP_STEPS)
            layers = []
            for l in range(SWEEP_LAYERS):
                c = synth.make_decode_case(base, 7000 + l, device=dev)
                layers.append(dict(q=c.q, k=c.k_pool, v=c.v_pool, pt=c.page_table, sl=c.seq_lens))
                del c
            g = torch.Generator(device=dev).manual_seed(99)
            k_new = torch.randn(SWEEP_STEPS, B, 8, 128, generator=g, device=dev).to(torch.bfloat16)
            v_new = torch.randn(SWEEP_STEPS, B, 8, 128, generator=g, device=dev).to(torch.bfloat16)
            lens = [torch.full((B,), ctx + s + 1, dtype=torch.int32, device=dev) for s in range(SWEEP_STEPS)]
            summ = None
            for bp in budgets:
                wl = synth.sweep_workload(B, ctx, bp, extra_tokens=SWEEP_STEPS)
                ks = synth.k_per_qhead(wl, ctx + SWEEP_STEPS)
                prob = sa.Problem(B=B, Hq=32, Hk=8, max_pages_per_seq=wl.max_pages_per_seq,
                                  num_pages=B * wl.max_pages_per_seq, sink=wl.S, window=wl.W,
                                  block_sizes=wl.block_sizes, k_per_head=ks, kcap=max(1, max(ks)),
                                  mode=sa.SUMMARY_MINMAX)
                ws = sa.Workspace(prob, device=dev)
                if summ is None:   # the prefill's summaries, one build per layer (budget-independent)
                    summ = []
                    for L in layers:
                        t = torch.empty(prob.summary_shape(), dtype=torch.bfloat16, device=dev)
                        sa.block_summarize(prob, L["k"], L["pt"], L["sl"], t, ws)
                        summ.append(t)
                idx = torch.empty(B, 32, prob.kcap, dtype=torch.int32, device=dev)
                cnt = torch.empty(B, 32, dtype=torch.int32, device=dev)
                out = torch.empty(B, 32, 128, device=dev)
                lse = torch.empty(B, 32, device=dev)

                def stack():
                    for s in range(SWEEP_STEPS):
                        for l, L in enumerate(layers):
                            sa.decode_step_append(prob, L["q"], k_new[s], v_new[s], L["k"], L["v"], L["pt"], lens[s],
                                                  summ[l], idx, cnt, out, lse, ws)

                with torch.cuda.stream(st):
                    stack()   # eager pass: kernel attributes, and the appended rows in place
                torch.cuda.synchronize()
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.stream(st):
                    with torch.cuda.graph(gr, stream=st, capture_error_mode="relaxed"):
                        stack()
                gr.replay()
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(st):
                    e0.record(st)
                    gr.replay()
                    e1.record(st)
                torch.cuda.synchronize()
                ms = e0.elapsed_time(e1)
                status = ws.status()
                # algorithmic bytes of the last layer-step (its selection), times the layer-steps
                nb = algorithmic_bytes(wl, prob, lens[-1].cpu().numpy(), idx, cnt)["total"]
                step_ms = ms / SWEEP_STEPS
                print(json.dumps({
                    "sweep_cell": {"batch": B, "context": ctx, "budget": bp / 10000, "layers": SWEEP_LAYERS,
                                   "steps": SWEEP_STEPS, "kv_gb": round(kv / 1e9, 1)},
                    "ms_per_token_step": round(step_ms, 4), "tokens_per_s": round(B / (step_ms / 1e3), 1),
                    "layer_queries_per_s": round(B * 32 * SWEEP_LAYERS / (step_ms / 1e3), 1),
                    "algorithmic_gb_per_s": round(nb * SWEEP_LAYERS / (step_ms / 1e3) / 1e9, 1),
                    "status": status}), flush=True)
                del gr, ws, idx, cnt
            del layers, summ, k_new, v_new
            torch.cuda.empty_cache()


def run_qwen(args, dev, rank, n_layers=4):
    """Config 2: the Qwen2.5-7B-shaped layer with head-specific granularity
    and budget (B16, 28 q / 4 KV heads, G = 7, ctx 65536, block size per KV
    head from {8, 16, 32, 64}, budget per KV head in [2 %, 20 %]; Fluxion core
    claim and Fig. 5): the whole step (sa_decode_step), `n_layers`
    independent layer copies (2.15 GB of KV each) rotating, a CUDA graph of K
    steps replayed R times."""
    wl = synth.workload("qwen_64k")
    ks = synth.k_per_qhead(wl)
    kcap = max(ks)
    prob = sa.Problem(B=wl.B, Hq=wl.Hq, Hk=wl.Hk, max_pages_per_seq=wl.max_pages_per_seq,
                      num_pages=wl.B * wl.max_pages_per_seq, sink=wl.S, window=wl.W,
                      block_sizes=wl.block_sizes, k_per_head=ks, kcap=kcap, mode=sa.SUMMARY_MINMAX)
    ws = sa.Workspace(prob, device=dev)
    layers = []
    for l in range(n_layers):
        c = synth.make_decode_case(wl, 1000 * rank + 2000 + l, device=dev)
        summ = torch.empty(prob.summary_shape(), dtype=torch.bfloat16, device=dev)
        sa.block_summarize(prob, c.k_pool, c.page_table, c.seq_lens, summ, ws)
        layers.append(dict(q=c.q, k=c.k_pool, v=c.v_pool, pt=c.page_table, sl=c.seq_lens, summ=summ,
                           sel_idx=torch.empty(wl.B, wl.Hq, kcap, dtype=torch.int32, device=dev),
                           sel_cnt=torch.empty(wl.B, wl.Hq, dtype=torch.int32, device=dev)))
        del c
    out = torch.empty(wl.B, wl.Hq, wl.D, device=dev)
    lse = torch.empty(wl.B, wl.Hq, device=dev)

    def step(L):
        sa.decode_step(prob, L["q"], L["k"], L["v"], L["pt"], L["sl"], L["summ"], L["sel_idx"], L["sel_cnt"], out,
                       lse, ws)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for L in layers:
            step(L)
    torch.cuda.synchronize()
    assert ws.status() == sa.SA_OK
    nbytes = [algorithmic_bytes(wl, prob, L["sl"].cpu().numpy(), L["sel_idx"], L["sel_cnt"])["total"]
              for L in layers]
    K, W = args.steps, args.warmup
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for i in range(W):
            step(layers[i % n_layers])
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for i in range(K):
                step(layers[(W + i) % n_layers])
    replay_ms(g, stream, 1)
    sp = spread(replay_ms(g, stream, args.repeats), K)
    ms = sp["median_ms_per_step"]
    b = float(np.mean([nbytes[(W + i) % n_layers] for i in range(K)]))
    peak, _ = measured_hbm_peak()
    achieved = b / (ms / 1e3) / 1e9
    assert ws.status() == sa.SA_OK
    del g, layers, ws
    torch.cuda.empty_cache()
    return {"workload": "qwen2.5-7b layer, decode, B16 x 28q/4kv heads (G 7) x D128, ctx 65536, block size per KV "
                        f"head {wl.block_sizes}, budget per KV head {[bp / 100 for bp in wl.budget_bp]} %, sinks 4, "
                        "window 1024, minmax summaries",
            "call": "sa_decode_step", "ms_per_step": ms, "spread": sp,
            "value": round(wl.B * wl.Hq / (ms / 1e3), 1), "unit": "queries/s",
            "algorithmic_bytes_per_step": int(b), "achieved": round(achieved, 1), "peak": peak, "unit_bw": "GB/s",
            "frac": round(achieved / peak, 4), "l2": f"{n_layers} rotating layer copies ({n_layers * 2.15:.1f} GB KV)"}


# --------------------------------------------------------------------------- oracle timing

def _bits(t):
    """bf16 tensor -> numpy uint16 bits on the host."""
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def _cell(name, unit, queries_per_step, secs_per_step, cores, sample, extrapolated):
    return {"cell": name, "value": round(queries_per_step / secs_per_step, 2), "unit": unit, "cores": cores,
            "s_per_step": round(secs_per_step, 4), "sample": sample, "extrapolated": extrapolated}


def _decode_cells(OT, pool, name, case_q, case_k, case_v, pt, lens, wl, ks, scale, budget_s, units=None,
                  total_units=None):
    """The oracle on one block-selection step of a case: one core (a bounded
    run over the units, scaled to the whole step when cut short) and all
    cores (every unit, or the sample `units` scaled to `total_units`)."""
    sp = OT.SharedPools(_bits(case_k), _bits(case_v))
    try:
        jobs = OT.decode_jobs(sp.spec(), case_q.float().cpu().numpy(), pt.cpu().numpy(), [int(x) for x in lens],
                              wl.block_sizes, ks, wl.S, wl.W, "minmax", scale, units=units)
        n_all = total_units or len(jobs)
        queries = wl.B * wl.Hq
        t1, n1 = OT.time_serial(jobs, sp.local, budget_s)
        one = _cell(name, "queries/s", queries, t1 / n1 * n_all, 1,
                    f"{n1} of {n_all} (sequence, KV head) units in {t1:.2f} s", n1 < n_all)
        tn = OT.time_parallel(pool, jobs)
        many = _cell(name, "queries/s", queries, tn * n_all / len(jobs), pool.cores,
                     f"{len(jobs)} of {n_all} units over {pool.cores} worker processes in {tn:.2f} s",
                     len(jobs) < n_all)
        return [one, many]
    finally:
        sp.close()


def cpu_baseline_cells(args, dev, L0, wl, ks, scale):
    """The oracle as it stands, timed on this machine's host cores on one
    core and on all of them (a spawn-started process pool over units), for
    the workloads of the hot path: the 4K tiny case, the 32K Llama layer
    (the headline), the 64K Qwen layer (a sampled slice, extrapolated), the
    128K score-table step (plus its 64-step total, extrapolated) and the
    batch-1 8K / 32K layers of the stack sweep."""
    from tests import oracle_timing as OT

    budget = max(2.0, args.cpu_seconds)
    pool = OT.OraclePool()
    cells = []
    try:
        # config 1: layer 0 of the headline run
        c1 = _decode_cells(OT, pool, "llama_32k: B8 x 32q/8kv, ctx 32768, 5 %", L0["q"], L0["k"], L0["v"], L0["pt"],
                           L0["sl"].tolist(), wl, ks, scale, budget * 0.4)
        cells += c1
        # config 0
        w0 = synth.workload("tiny_4k")
        c = synth.make_decode_case(w0, 0, device=dev)
        cells += _decode_cells(OT, pool, "tiny_4k: B1 x 8q/2kv, ctx 4096, 10 %", c.q, c.k_pool, c.v_pool,
                               c.page_table, c.seq_lens.tolist(), w0, synth.k_per_qhead(w0), scale, budget * 0.05)
        # config 4: batch-1 cells of the sweep, one layer, 5 % budget
        for ctx in (8192, 32768):
            w4 = synth.sweep_workload(1, ctx, 500, extra_tokens=0)
            c = synth.make_decode_case(w4, 7000, device=dev)
            cells += _decode_cells(OT, pool, f"stack sweep cell: B1 x 32q/8kv, ctx {ctx}, 5 %, one layer", c.q,
                                   c.k_pool, c.v_pool, c.page_table, c.seq_lens.tolist(), w4,
                                   synth.k_per_qhead(w4), scale, budget * 0.05)
        # config 2: one unit per KV head on one core, 16 units over the pool; scaled to the 64 units
        w2 = synth.workload("qwen_64k")
        c = synth.make_decode_case(w2, 2000, device=dev)
        units = [(b, b % w2.Hk) for b in range(w2.B)]   # every KV head (block size, budget) four times
        cells += _decode_cells(OT, pool, "qwen_64k: B16 x 28q/4kv, ctx 65536, per-KV-head Bs and budget", c.q,
                               c.k_pool, c.v_pool, c.page_table, c.seq_lens.tolist(), w2, synth.k_per_qhead(w2),
                               scale, budget * 0.15, units=units, total_units=w2.B * w2.Hk)
        del c
        # config 3: one score-table step, every head; the 64-step total scaled from it
        w3 = synth.table_workload("tables_128k")
        tc = synth.make_table_case(w3, 7, device=dev)
        sp = OT.SharedPools(_bits(tc.k_pool), _bits(tc.v_pool))
        try:
            heads = [(b, h) for b in range(w3.B) for h in range(w3.Hq)]
            jobs = OT.table_jobs(sp.spec(), tc.q_steps[0].float().cpu().numpy(), tc.q_steps[1].float().cpu().numpy(),
                                 tc.page_table.cpu().numpy(), tc.vert0.cpu().numpy(), tc.slash0.cpu().numpy(), w3.L0,
                                 w3.S, w3.W, w3.beta, w3.kcap, w3.G, scale, heads)
            t1, n1 = OT.time_serial(jobs, sp.local, budget * 0.3)
            q3 = w3.B * w3.Hq
            name = "tables_128k: B4 x 32q/8kv, ctx 131072 + 1, score-table step"
            one = _cell(name, "queries/s", q3, t1 / n1 * len(jobs), 1, f"{n1} of {len(jobs)} heads in {t1:.2f} s",
                        n1 < len(jobs))
            tn = OT.time_parallel(pool, jobs)
            many = _cell(name, "queries/s", q3, tn, pool.cores, f"{len(jobs)} heads over {pool.cores} workers", False)
            for cc in (one, many):
                cc["s_per_64_steps"] = round(cc["s_per_step"] * w3.steps, 2)
                cc["s_per_64_steps_extrapolated"] = True
            cells += [one, many]
        finally:
            sp.close()
        del tc
        torch.cuda.empty_cache()
    finally:
        pool.close()
    head = c1[1]
    return {"value": head["value"], "unit": "queries/s", "cores": head["cores"], "kind": "oracle",
            "sample": f"llama_32k step, {head['sample']}; one core: {c1[0]['value']} queries/s ({c1[0]['sample']})",
            "cells": cells}


def run_reference(args):
    """The reference arm: the oracle as it stands on this machine's host
    cores (a spawn-started process pool over the (sequence, KV head) units),
    one whole 32K Llama-layer step per timed step; inputs generated on the
    host, no GPU."""
    world, rank, local = dist_info()
    if rank != 0:
        return
    from tests import oracle_timing as OT

    wl = synth.workload(WORKLOAD)
    ks = synth.k_per_qhead(wl)
    c = synth.make_decode_case(wl, 100)
    sp = OT.SharedPools(_bits(c.k_pool), _bits(c.v_pool))
    pool = OT.OraclePool()
    try:
        jobs = OT.decode_jobs(sp.spec(), c.q.float().numpy(), c.page_table.numpy(), c.seq_lens.tolist(),
                              wl.block_sizes, ks, wl.S, wl.W, "minmax", 1 / math.sqrt(wl.D))
        # a step is the whole layer step when the pool can do it in about a second, else a bounded
        # sample of its units (scaled to queries of the units done)
        per_step = max(1, min(len(jobs), int(len(jobs) * pool.cores / 16)))
        for i in range(args.warmup):
            OT.time_parallel(pool, jobs[:pool.cores])
        t0 = time.perf_counter()
        for i in range(args.steps):
            OT.time_parallel(pool, jobs[:per_step])
        dt = time.perf_counter() - t0
    finally:
        pool.close()
        sp.close()
    nq = per_step * wl.G * args.steps
    v = round(nq / dt, 2)
    sample = (f"{per_step} of {len(jobs)} (sequence, KV head) units of one 32K Llama-layer step per timed step "
              f"(summaries + canonical scores + top-k + fp64 attention + merge), {args.steps} steps, "
              f"{pool.cores} worker processes")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "queries/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V with planted sink, heavy blocks and recency ramp)",
        "config": headline_config(world),
        "cpu_baseline": {"value": v, "unit": "queries/s", "cores": pool.cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "queries/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=N_LAYERS,
                    help="independent layer copies rotated per step (1.07 GB of KV each)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-tables", action="store_true", help="skip the score-table (a7) leg")
    ap.add_argument("--no-group", action="store_true", help="skip the group-shared selection variant")
    ap.add_argument("--no-bypass", action="store_true", help="skip the head-sparsity bypass variant")
    ap.add_argument("--no-config2", action="store_true", help="skip the Qwen-shaped 64K leg (config 2)")
    ap.add_argument("--repeats", type=int, default=30, help="replays of each timed CUDA graph (median, p10, p90)")
    ap.add_argument("--sweep", action="store_true",
                    help="the batch x context x budget throughput sweep of a 32-layer stack (one line per cell)")
    ap.add_argument("--sweep-cells", default="",
                    help="with --sweep: only these cells, as batch:context:budget_bp[,...]")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.sweep:
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
