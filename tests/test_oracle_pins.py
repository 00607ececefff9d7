"""Pins of the fp64 oracle to facts that do not come from the oracle itself:
closed forms, library routines on special cases, hand-worked values,
invariants of the method and brute force on tiny inputs."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import sparse_attention_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def rand_bf16(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(F32)
    return torch.from_numpy(x).to(torch.bfloat16).float().numpy()


# ---------------------------------------------------------------- bf16 rounding

def test_bf16_rne_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200_000).astype(F32) * F32(3.0)
    # exact ties: low 16 bits == 0x8000, with even and odd kept parts
    ties = (rng.integers(0x3F000000, 0x40800000, 4096, dtype=np.int64) & ~0xFFFF | 0x8000).astype(np.uint32)
    x = np.concatenate([x, ties.view(F32), -ties.view(F32), np.array([0.0, -0.0, 1.0, 65504.0], F32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    got = orc.bf16_rne(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# ---------------------------------------------------------------- partition

@pytest.mark.parametrize("L,S,W,Bs,ncand", [
    (4096, 4, 256, 16, 240),        # tiny 4K workload: 10 % budget -> 24 blocks
    (32768, 4, 1024, 16, 1984),     # Llama-shaped 32K workload: 5 % -> 100 blocks
    (65536, 4, 1024, 8, 8064),
    (65536, 4, 1024, 16, 4032),
    (65536, 4, 1024, 32, 2016),
    (65536, 4, 1024, 64, 1008),
    (1000, 4, 996, 16, 0),          # sinks + window cover the context
    (0, 4, 1024, 16, 0),
])
def test_candidate_counts(L, S, W, Bs, ncand):
    j0, j1 = orc.candidate_blocks(L, S, W, Bs)
    assert j1 - j0 == ncand


def test_partition_is_disjoint_cover():
    for L, S, W, Bs in [(100, 4, 16, 16), (37, 4, 16, 8), (5, 4, 16, 16), (300, 7, 64, 64)]:
        I = orc.dense_tokens(L, S, W)
        j0, j1 = orc.candidate_blocks(L, S, W, Bs)
        J = orc.sparse_tokens(L, S, W, Bs, range(j0, j1))
        both = np.concatenate([I, J])
        assert len(np.unique(both)) == len(both) == L
        assert set(both.tolist()) == set(range(L))


# ---------------------------------------------------------------- canonical score order

def test_canonical_dot_exact_on_small_integers():
    # every partial sum is an integer below 2^24 -> any order is exact
    rng = np.random.default_rng(1)
    q = rng.integers(-16, 17, 128).astype(F32)
    x = rng.integers(-64, 65, (500, 128)).astype(F32)
    got = orc.canonical_dot(q, x)
    ref = (x.astype(np.int64) * q.astype(np.int64)[None, :]).sum(axis=1)
    assert np.array_equal(got.astype(np.int64), ref)


def test_canonical_dot_handworked_order():
    cases = json.load(open(os.path.join(GOLDEN, "canonical_score_cases.json")))["cases"]
    for c in cases:
        q = np.zeros(128, F32)
        x = np.zeros((1, 128), F32)
        for d, qv, xv in c["terms"]:
            q[d] = qv
            x[0, d] = xv
        assert float(orc.canonical_dot(q, x)[0]) == c["expected"], c["name"]


def test_canonical_dot_close_to_fp64():
    rng = np.random.default_rng(2)
    q = rand_bf16(rng, 128)
    x = rand_bf16(rng, (300, 128))
    got = orc.canonical_dot(q, x).astype(np.float64)
    exact = (x.astype(np.float64) * q.astype(np.float64)).sum(axis=1)
    bound = 20 * 2.0 ** -24 * (np.abs(x) * np.abs(q)).sum(axis=1)   # <= 18 roundings per path
    assert np.all(np.abs(got - exact) <= bound)


def test_canonical_dot_negative_zero_becomes_positive():
    q = np.zeros(128, F32)
    q[0] = -1.0
    x = np.zeros((1, 128), F32)
    out = orc.canonical_dot(q, x)
    assert out[0] == 0 and not np.signbit(out[0])


# ---------------------------------------------------------------- summaries

def test_minmax_summary_and_bound():
    rng = np.random.default_rng(3)
    for Bs in (8, 16, 32, 64):
        keys = rand_bf16(rng, (Bs, 128))
        s = orc.summarize_block(keys, orc.SUMMARY_MINMAX)
        assert np.array_equal(s[0], keys.min(axis=0)) and np.array_equal(s[1], keys.max(axis=0))
        for _ in range(20):
            q = rand_bf16(rng, 128)
            sc = float(orc.score_blocks(q, s[None], orc.SUMMARY_MINMAX)[0])
            best = float((keys.astype(np.float64) @ q.astype(np.float64)).max())
            assert sc >= best - 1e-4 * (1 + abs(best))
            # the select form equals sum_d max(q kmax, q kmin)
            alt = np.maximum(q * s[1], q * s[0]).astype(np.float64).sum()
            assert abs(sc - alt) <= 1e-4 * (1 + abs(alt))


def test_mean_summary_exact_case_matches_library_rounding():
    # keys on a grid of 2^-6: fp32 sums are exact, the division by a power of
    # two is exact, so the summary is the library bf16 rounding of the true mean
    rng = np.random.default_rng(4)
    for Bs in (8, 16, 32, 64):
        keys = (rng.integers(-300, 301, (Bs, 128)) / 64.0).astype(F32)
        s = orc.summarize_block(keys, orc.SUMMARY_MEAN)
        true_mean = keys.astype(np.float64).sum(axis=0) / Bs
        ref = torch.from_numpy(true_mean.astype(F32)).to(torch.bfloat16).float().numpy()
        assert np.array_equal(s, ref)


def test_mean_summary_random_close():
    rng = np.random.default_rng(5)
    keys = rand_bf16(rng, (16, 128))
    s = orc.summarize_block(keys, orc.SUMMARY_MEAN).astype(np.float64)
    true_mean = keys.astype(np.float64).mean(axis=0)
    assert np.all(np.abs(s - true_mean) <= 2.0 ** -8 * np.abs(true_mean) + 1e-6)


def test_mean_score_times_block_equals_sum_of_dots():
    # Bs * (q . mean_k) == sum_t q . k_t  (fp64, before any rounding)
    rng = np.random.default_rng(6)
    keys = rand_bf16(rng, (32, 128)).astype(np.float64)
    q = rand_bf16(rng, 128).astype(np.float64)
    lhs = 32 * (q @ keys.mean(axis=0))
    rhs = (keys @ q).sum()
    assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


# ---------------------------------------------------------------- top-k

def _selection_property(scores, ids, sel):
    chosen = set(sel.tolist())
    for a in range(len(ids)):
        for b in range(len(ids)):
            if ids[a] in chosen and ids[b] not in chosen:
                if not (scores[a] > scores[b] or (scores[a] == scores[b] and ids[a] < ids[b])):
                    return False
    return True


def test_topk_brute_force_small():
    rng = np.random.default_rng(7)
    for trial in range(60):
        n = int(rng.integers(1, 13))
        scores = rng.integers(-3, 4, n).astype(F32)          # many ties
        ids = np.arange(n) + int(rng.integers(0, 5))
        for k in range(0, n + 2):
            sel = orc.topk_blocks(scores, ids, k)
            assert len(sel) == min(k, n)
            assert np.all(np.diff(sel) > 0)
            assert _selection_property(scores, ids, sel)
            # brute force: the best k-subset in (score desc, index asc) order
            kk = min(k, n)
            best = None
            for sub in itertools.combinations(range(n), kk):
                key = sorted(((-scores[i], ids[i]) for i in sub))
                if best is None or key < best[0]:
                    best = (key, sub)
            assert sorted(ids[list(best[1])].tolist()) == sel.tolist()


def test_topk_all_equal_takes_lowest_indices():
    ids = np.arange(10, 50)
    sel = orc.topk_blocks(np.full(40, 1.5, F32), ids, 7)
    assert sel.tolist() == list(range(10, 17))


# ---------------------------------------------------------------- attention and merge

def _torch_sdpa(q, K, V, scale):
    qt = torch.from_numpy(np.asarray(q, np.float64)).reshape(1, 1, 1, -1)
    Kt = torch.from_numpy(np.asarray(K, np.float64)).reshape(1, 1, K.shape[0], -1)
    Vt = torch.from_numpy(np.asarray(V, np.float64)).reshape(1, 1, V.shape[0], -1)
    O = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale).reshape(-1).numpy()
    lse = torch.logsumexp(scale * (Kt.reshape(K.shape[0], -1) @ qt.reshape(-1)), dim=0).item()
    return O, lse


def test_attend_matches_torch_sdpa():
    rng = np.random.default_rng(8)
    for n in (1, 2, 17, 300):
        K = rand_bf16(rng, (n, 128))
        V = rand_bf16(rng, (n, 128))
        q = rand_bf16(rng, 128)
        O, lse = orc.attend(q, K, V, np.arange(n), 1 / math.sqrt(128))
        O_ref, lse_ref = _torch_sdpa(q, K, V, 1 / math.sqrt(128))
        assert np.max(np.abs(O - O_ref)) < 1e-12 and abs(lse - lse_ref) < 1e-12


def test_single_token_attention():
    rng = np.random.default_rng(9)
    K = rand_bf16(rng, (5, 128))
    V = rand_bf16(rng, (5, 128))
    q = rand_bf16(rng, 128)
    O, lse = orc.attend(q, K, V, np.array([3]), 0.25)
    assert np.array_equal(O, V[3].astype(np.float64))
    assert abs(lse - 0.25 * float(K[3].astype(np.float64) @ q.astype(np.float64))) < 1e-12


def test_lse_identity_on_random_partitions():
    rng = np.random.default_rng(10)
    n = 400
    K = rand_bf16(rng, (n, 128), 2.0)
    V = rand_bf16(rng, (n, 128))
    q = rand_bf16(rng, 128)
    sc = 1 / math.sqrt(128)
    O_all, lse_all = orc.attend(q, K, V, np.arange(n), sc)
    for parts in (2, 3, 5):
        lab = rng.integers(0, parts, n)
        O, lse = orc.attend(q, K, V, np.nonzero(lab == 0)[0], sc)
        for p in range(1, parts):
            Op, lp = orc.attend(q, K, V, np.nonzero(lab == p)[0], sc)
            O, lse = orc.lse_merge(O, lse, Op, lp)
        assert np.max(np.abs(O - O_all)) < 1e-12 and abs(lse - lse_all) < 1e-12


def test_lse_merge_with_empty_side():
    O = np.arange(128, dtype=np.float64)
    Om, lm = orc.lse_merge(O, 1.25, np.zeros(128), -math.inf)
    assert np.array_equal(Om, O) and lm == 1.25
    Om, lm = orc.lse_merge(np.zeros(128), -math.inf, np.zeros(128), -math.inf)
    assert np.all(Om == 0) and lm == -math.inf


# ---------------------------------------------------------------- paged gather

def test_gather_sequence_inverts_page_scatter():
    rng = np.random.default_rng(11)
    P, Hk, D, npg = 16, 3, 128, 9
    L = npg * P - 5
    logical = rng.standard_normal((Hk, npg * P, D)).astype(F32)
    perm = rng.permutation(npg + 4)[:npg]
    pool = np.zeros((npg + 4, Hk, P, D), F32)
    for lp in range(npg):
        for h in range(Hk):
            pool[perm[lp], h] = logical[h, lp * P:(lp + 1) * P]
    for h in range(Hk):
        assert np.array_equal(orc.gather_sequence(pool, perm, h, L), logical[h, :L])


# ---------------------------------------------------------------- whole-step special cases

def _case(rng, L, Bs=16, S=4, W=64):
    K = rand_bf16(rng, (L, 128))
    V = rand_bf16(rng, (L, 128))
    q = rand_bf16(rng, 128)
    return q, K, V


def test_full_budget_reproduces_dense_attention():
    rng = np.random.default_rng(12)
    for L, Bs in ((1000, 16), (777, 8), (2048, 64)):
        q, K, V = _case(rng, L)
        j0, j1 = orc.candidate_blocks(L, 4, 64, Bs)
        sel, _, _ = orc.select_head(q, K, L, 4, 64, Bs, j1 - j0, orc.SUMMARY_MINMAX)
        r = orc.decode_head(q, K, V, L, 4, 64, Bs, sel, 1 / math.sqrt(128))
        O_ref, lse_ref = _torch_sdpa(q, K[:L], V[:L], 1 / math.sqrt(128))
        assert np.max(np.abs(r["O"] - O_ref)) < 1e-12 and abs(r["lse"] - lse_ref) < 1e-12


def test_window_covering_context_is_dense():
    rng = np.random.default_rng(13)
    L = 60
    q, K, V = _case(rng, L)
    sel, ids, _ = orc.select_head(q, K, L, 4, 64, 16, 3, orc.SUMMARY_MEAN)
    assert len(ids) == 0 and len(sel) == 0
    r = orc.decode_head(q, K, V, L, 4, 64, 16, sel, 0.1)
    O_ref, lse_ref = _torch_sdpa(q, K, V, 0.1)
    assert np.max(np.abs(r["O"] - O_ref)) < 1e-12 and len(r["J"]) == 0


def test_zero_budget_is_dense_part_only():
    rng = np.random.default_rng(14)
    L = 900
    q, K, V = _case(rng, L)
    sel, _, _ = orc.select_head(q, K, L, 4, 64, 16, 0, orc.SUMMARY_MINMAX)
    r = orc.decode_head(q, K, V, L, 4, 64, 16, sel, 0.1)
    I = np.concatenate([np.arange(4), np.arange(L - 64, L)])
    O_ref, lse_ref = _torch_sdpa(q, K[I], V[I], 0.1)
    assert len(sel) == 0 and np.max(np.abs(r["O"] - O_ref)) < 1e-12


def test_selected_block_contributes_only_its_middle_tokens():
    # block 0 holds the sinks; a selected block straddling the window start
    # contributes only the tokens before the window
    L, S, W, Bs = 200, 4, 40, 16
    J = orc.sparse_tokens(L, S, W, Bs, [0, 9])
    assert J.tolist() == list(range(4, 16)) + list(range(144, 160))
    J2 = orc.sparse_tokens(195, S, W, Bs, [9])       # window starts at 155
    assert J2.tolist() == list(range(144, 155))


def test_planted_heavy_block_is_selected():
    # a block whose keys all get + c * q_dir must win the top-1 (both summaries)
    rng = np.random.default_rng(15)
    L, Bs = 1024, 16
    q, K, V = _case(rng, L)
    qd = q / np.linalg.norm(q) * math.sqrt(128)
    K2 = K.copy()
    K2[37 * Bs:38 * Bs] = torch.from_numpy((K2[37 * Bs:38 * Bs] + 1.5 * qd).astype(F32)).to(torch.bfloat16).float().numpy()
    for mode in (orc.SUMMARY_MINMAX, orc.SUMMARY_MEAN):
        sel, _, _ = orc.select_head(q, K2, L, 4, 64, Bs, 1, mode)
        assert sel.tolist() == [37]


def test_empty_sequence():
    q = np.ones(128, F32)
    K = np.zeros((0, 128), F32)
    r = orc.decode_head(q, K, K, 0, 4, 64, 16, [], 0.1)
    assert np.all(r["O"] == 0) and r["lse"] == -math.inf


# ---------------------------------------------------------------------------
# variant: group-shared selection (reading R9)
# ---------------------------------------------------------------------------

def _group_case(seed, G, n_blocks, Bs=16, D=128):
    rng = np.random.default_rng(seed)
    L = n_blocks * Bs
    kseq = orc.bf16_rne(rng.standard_normal((L, D)).astype(np.float32))
    qs = [orc.bf16_rne(rng.standard_normal(D).astype(np.float32)) for _ in range(G)]
    return qs, kseq, L


def test_group_selection_of_one_head_is_the_head_selection():
    qs, kseq, L = _group_case(1, 1, 40)
    for mode in (orc.SUMMARY_MINMAX, orc.SUMMARY_MEAN):
        for k in (0, 1, 5, 17, 39):
            a, _, _ = orc.select_head(qs[0], kseq, L, 0, 16, 16, k, mode)
            b, _, _ = orc.select_group(qs, kseq, L, 0, 16, 16, k, mode)
            assert np.array_equal(a, b)


def test_group_selection_maximises_the_group_score_sum():
    # brute force over every k-subset of a small candidate range: the chosen
    # blocks carry the largest total group score (exact fp64 sums of the fp32
    # group scores; with distinct scores the optimum is unique)
    import itertools
    for seed in range(4):
        qs, kseq, L = _group_case(10 + seed, 3, 12)
        for k in (1, 2, 4, 6):
            sel, ids, sc = orc.select_group(qs, kseq, L, 0, 16, 16, k, orc.SUMMARY_MINMAX)
            assert len(np.unique(sc)) == len(sc)
            best = max(itertools.combinations(range(len(ids)), k), key=lambda c: sum(float(sc[i]) for i in c))
            assert np.array_equal(sel, np.sort(ids[list(best)]))


def test_group_sum_can_overrule_a_single_head():
    # a block one head likes strongly but the other three dislike is kept by
    # that head alone, and dropped by the group when the others' dislike wins
    D, Bs, n = 128, 16, 20
    rng = np.random.default_rng(7)
    base = rng.standard_normal((n * Bs, D)).astype(np.float32) * 0.05
    u = np.zeros(D, np.float32); u[0] = 1.0
    w = np.zeros(D, np.float32); w[1] = 1.0
    kseq = base.copy()
    kseq[5 * Bs:6 * Bs] += 4.0 * u          # block 5: along u
    kseq[9 * Bs:10 * Bs] += 1.0 * w         # block 9: mildly along w
    kseq = orc.bf16_rne(kseq)
    q_like = orc.bf16_rne((8.0 * u + 0.5 * w).astype(np.float32))
    q_dis = orc.bf16_rne((-8.0 * u + 2.0 * w).astype(np.float32))
    qs = [q_like, q_dis, q_dis, q_dis]
    own, _, _ = orc.select_head(q_like, kseq, n * Bs, 0, 16, Bs, 1, orc.SUMMARY_MEAN)
    grp, _, sc = orc.select_group(qs, kseq, n * Bs, 0, 16, Bs, 1, orc.SUMMARY_MEAN)
    assert own.tolist() == [5]
    assert grp.tolist() == [9]


# ---------------------------------------------------------------------------
# exact top-k inside the table candidates (reading R10)
# ---------------------------------------------------------------------------

def test_exact_token_topk_against_full_sort():
    # brute force: the kept set is the k best of a full fp64 sort of the exact
    # dot products (distinct scores), for every k
    rng = np.random.default_rng(21)
    D, L = 128, 300
    kseq = orc.bf16_rne(rng.standard_normal((L, D)).astype(np.float32))
    q = orc.bf16_rne(rng.standard_normal(D).astype(np.float32))
    cand = np.sort(rng.choice(L, 40, replace=False))
    exact = kseq[cand].astype(np.float64) @ q.astype(np.float64)
    for k in range(0, 42, 3):
        kept, sc = orc.exact_token_topk(q, kseq, cand, k)
        assert len(sc) == len(cand)
        want = np.sort(cand[np.argsort(-exact, kind="stable")[:min(k, len(cand))]])
        assert np.array_equal(kept, want)


def test_exact_token_topk_edge_cases():
    rng = np.random.default_rng(22)
    kseq = orc.bf16_rne(rng.standard_normal((64, 128)).astype(np.float32))
    q = orc.bf16_rne(rng.standard_normal(128).astype(np.float32))
    kept, sc = orc.exact_token_topk(q, kseq, np.zeros(0, np.int64), 5)
    assert len(kept) == 0 and len(sc) == 0
    cand = np.array([3, 9, 17])
    kept, _ = orc.exact_token_topk(q, kseq, cand, 10)      # k beyond the list keeps it whole
    assert kept.tolist() == [3, 9, 17]
    # equal keys score equally: the lower position wins the tie
    kdup = kseq.copy()
    kdup[40] = kdup[7]
    kept, sc = orc.exact_token_topk(q, kdup, np.array([7, 40]), 1)
    assert sc[0] == sc[1] and kept.tolist() == [7]
