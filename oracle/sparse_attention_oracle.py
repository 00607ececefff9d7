"""fp64 CPU oracle for decode-phase hybrid sparse attention over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module.  It shares no code with the
CUDA path: it is a plain, slow restatement of what the method computes, written
with numpy so that a reader can check each step against the pages by eye.

Precision: block selection (summaries, block scores, top-k) runs in a fixed
canonical fp32 order, because an fp32 decision made on both sides in the same
precision is what lets index sets match bit for bit; attention, the
log-sum-exp merge and the score-table updates run in fp64.

Sources (page title, section / equation / figure):
  * "HGCA: Hybrid GPU-CPU Attention for Long Context LLM Inference", review
    section "What carries the argument": dense attention over a recent window
    and sparse attention over selected older entries, merged by the exact
    log-sum-exp identity O = (e^lse_I O_I + e^lse_J O_J) / (e^lse_I + e^lse_J),
    lse_S = log sum_{j in S} e^{s_j}; minor comment on Sec. 3.3 (stabilise the
    merge by the maximum); the moving average of attention weights (MAW) and the
    per-head threshold beta / (number of GPU-side entries).
  * "An Efficient Hybrid Sparse Attention with CPU-GPU Parallelism for
    Long-Context Inference" (Fluxion), core claim and Fig. 2 / Fig. 5: block
    top-k selection with a head-specific block size and budget; Fig. 4: the
    attention sink.
  * "Unifying Sparse Attention with Hierarchical Memory for Scalable
    Long-Context LLM Serving" (SPIN), abstract and Fig. 6: the paged KV
    substrate reached through a page table.
  * "Learn from the Past: Fast Sparse Indexing for Large Language Model
    Decoding" (LFPS), "What carries the argument", Eq. (9), Eq. (10): vertical
    and slash score tables with decay r = 0.95 and positional expansion by
    offsets {-1, 0, 1, 2}; Algorithm 1 step 1, Eq. (5), Eq. (6), App. B.1
    ("Assumptions & free parameters"): the head-sparsity estimate and the
    mean-value bypass with epsilon = 0.85.

Readings where the pages are silent (each also listed in the design notes):
  R1  I = sinks [0, min(S, L)) U window [max(L - W, min(S, L)), L);
      M = the tokens between them.  Candidate blocks are the blocks that meet M;
      a selected block contributes only its tokens in M, so I and J are disjoint.
  R2  The budget is an integer k per query head given by the caller.
  R3  MINMAX summary: per-dimension min and max of the block's bf16 keys; block
      score s = sum_d q_d * (q_d >= 0 ? kmax_d : kmin_d) (the bounding-box upper
      bound of max_t q.k_t).  MEAN summary: bf16(RNE(fp32 sum over the block's
      tokens in ascending order / n)).  The pages never define either.
  R4  Canonical fp32 score order: the 128 dims are split into 8 lanes of 16
      consecutive dims; each lane sums its products in ascending dim order with
      one rounding per step; the 8 lane sums are combined by a butterfly with
      partner offsets 4, 2, 1.  Result + 0.0 (turns -0 into +0).
  R5  Top-k order: score descending, block index ascending; report ascending.
  R6  Score tables: EMA  T <- r T + (1 - r) a  with a the merged softmax
      weight (0 for unattended entries); vertical indexed by absolute position,
      slash by offset (L - 1 - i); one threshold tau = beta / |I|, strict
      comparison; expansion {-1, 0, 1, 2} clipped to M; at most kcap tokens
      (lowest positions kept).
  R9  Group-shared selection (a variant; the pages select per head): the
      blocks of a KV head are ranked by the fp32 sum, in head order, of its G
      query heads' canonical scores; every head of the group keeps the same k
      blocks (ties by lower block index).
  R10 Exact top-k inside the table candidates (LFPS, "The reading": an exact
      top-k needs a dot product against every key; the tables only narrow the
      keys down): each candidate token's score is the canonical fp32 dot
      product of q with its bf16 key row (reading R4's order), and the k best
      by (score descending, position ascending) are kept, reported ascending.
  R11 Head-sparsity bypass (LFPS Algorithm 1 step 1, Eq. (5), Eq. (6),
      App. B.1; epsilon = 0.85): tokens split into the sink (token 0), the
      local window (the six newest of the L keys) and the n global tokens
      between; the global mass is n times the log-normal mean of e^z with the
      page's sigma^2 read as the keys' mean per-dimension variance times the
      softmax scale squared.  rho = sink mass / total; rho > epsilon bypasses
      the head: output the mean value row over all L tokens, lse = log of the
      total mass, and the head's score tables skip the next update.
"""
from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64

SUMMARY_MINMAX = "minmax"
SUMMARY_MEAN = "mean"


# ---------------------------------------------------------------------------
# bf16 rounding (round to nearest, ties to even) of float32 values
# ---------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """Round float32 values to the nearest bf16 value (ties to even), returned
    as float32.  Finite inputs only (the summaries never overflow)."""
    a = np.ascontiguousarray(np.asarray(x, dtype=F32))
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    return r.astype(np.uint32).view(F32).reshape(a.shape)


# ---------------------------------------------------------------------------
# partition of the context into dense and sparse parts (reading R1)
# ---------------------------------------------------------------------------

def partition(L: int, S: int, W: int):
    """Return (s_end, w_beg): I = [0, s_end) U [w_beg, L), M = [s_end, w_beg).

    HGCA review, "What carries the argument": the recent window is attended
    densely; Fluxion Fig. 4: the sink tokens carry large attention and are
    kept."""
    s_end = min(S, L)
    w_beg = max(L - W, s_end)
    return s_end, w_beg


def dense_tokens(L: int, S: int, W: int) -> np.ndarray:
    s_end, w_beg = partition(L, S, W)
    return np.concatenate([np.arange(0, s_end), np.arange(w_beg, L)]).astype(np.int64)


def candidate_blocks(L: int, S: int, W: int, Bs: int):
    """Blocks that meet M: j in [s_end // Bs, ceil(w_beg / Bs)), empty if M is."""
    s_end, w_beg = partition(L, S, W)
    if w_beg <= s_end:
        return 0, 0
    return s_end // Bs, -(-w_beg // Bs)


def sparse_tokens(L: int, S: int, W: int, Bs: int, blocks) -> np.ndarray:
    """J = (union of the selected blocks' tokens) intersected with M."""
    s_end, w_beg = partition(L, S, W)
    toks = []
    for j in sorted(set(int(x) for x in blocks)):
        lo, hi = max(j * Bs, s_end), min((j + 1) * Bs, w_beg)
        if lo < hi:
            toks.append(np.arange(lo, hi))
    if not toks:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate(toks).astype(np.int64)


# ---------------------------------------------------------------------------
# paged KV gather (SPIN abstract / Fig. 6: KV lives in fixed-size pages)
# ---------------------------------------------------------------------------

def gather_sequence(pool: np.ndarray, page_row: np.ndarray, kvh: int, L: int) -> np.ndarray:
    """Logical [L, D] rows of one (sequence, KV head) from a pool laid out
    [num_pages][Hk][P][D]: token t lives in page page_row[t // P], row t % P."""
    P = pool.shape[2]
    t = np.arange(L)
    return pool[page_row[t // P], kvh, t % P, :]


# ---------------------------------------------------------------------------
# step a1: block summaries (reading R3)
# ---------------------------------------------------------------------------

def summarize_block(keys: np.ndarray, mode: str) -> np.ndarray:
    """Summary of one block given its keys [n, D] (bf16 values held in float32).

    MINMAX -> [2, D] (row 0 = min, row 1 = max), exact.
    MEAN   -> [D]: fp32 running sum in ascending token order, IEEE fp32 division
              by n, then round-to-nearest-even to bf16."""
    keys = np.asarray(keys, dtype=F32)
    if mode == SUMMARY_MINMAX:
        return np.stack([keys.min(axis=0), keys.max(axis=0)])
    acc = keys[0].copy()
    for t in range(1, keys.shape[0]):
        acc = (acc + keys[t]).astype(F32)
    return bf16_rne((acc / F32(keys.shape[0])).astype(F32))


def summarize_sequence(kseq: np.ndarray, Bs: int, mode: str, j_begin: int = 0, j_end=None):
    """Summaries of blocks [j_begin, j_end) of one sequence; block j covers
    tokens [j Bs, min((j+1) Bs, L)).  Returns [n, 2, D] or [n, D] float32."""
    L = kseq.shape[0]
    if j_end is None:
        j_end = -(-L // Bs)
    out = [summarize_block(kseq[j * Bs:min((j + 1) * Bs, L)], mode) for j in range(j_begin, j_end)]
    D = kseq.shape[1]
    if not out:
        return np.zeros((0, 2, D) if mode == SUMMARY_MINMAX else (0, D), dtype=F32)
    return np.stack(out)


# ---------------------------------------------------------------------------
# step a2: block scores in the canonical fp32 order (readings R3, R4)
# ---------------------------------------------------------------------------

def summary_operand(q32: np.ndarray, summ: np.ndarray, mode: str) -> np.ndarray:
    """The per-dim key values the score multiplies q by: [n, D]."""
    if mode == SUMMARY_MINMAX:
        return np.where(q32[None, :] >= 0, summ[:, 1, :], summ[:, 0, :]).astype(F32)
    return summ.astype(F32)


def canonical_dot(q32: np.ndarray, x: np.ndarray) -> np.ndarray:
    """sum_d q_d x_d for each row of x [n, 128] in the canonical fp32 order:
    8 lanes x 16 consecutive dims summed in ascending order, then a butterfly
    over lane partners at offsets 4, 2, 1; finally + 0.0."""
    n, D = x.shape
    assert D == 128
    prod = (x * q32[None, :]).astype(F32)           # exact: bf16 x bf16 fits fp32
    lanes = prod.reshape(n, 8, 16)
    acc = lanes[:, :, 0].copy()
    for i in range(1, 16):
        acc = (acc + lanes[:, :, i]).astype(F32)
    lane = np.arange(8)
    for off in (4, 2, 1):
        acc = (acc + acc[:, lane ^ off]).astype(F32)
    return (acc[:, 0] + F32(0.0)).astype(F32)


def score_blocks(q32: np.ndarray, summ: np.ndarray, mode: str) -> np.ndarray:
    """Block scores of one query head against n block summaries (unscaled: the
    softmax scale is positive and does not change the ranking)."""
    return canonical_dot(np.asarray(q32, dtype=F32), summary_operand(q32, summ, mode))


# ---------------------------------------------------------------------------
# step a3: per-head top-k (reading R5)
# ---------------------------------------------------------------------------

def topk_blocks(scores: np.ndarray, block_ids: np.ndarray, k: int) -> np.ndarray:
    """Keep the k best blocks by (score descending, block index ascending) and
    return their indices in ascending order.  Fluxion core claim: each head
    keeps its own top-k block set."""
    n = len(block_ids)
    k = max(0, min(int(k), n))
    if k == 0:
        return np.zeros(0, dtype=np.int64)
    if k == n:
        return np.sort(np.asarray(block_ids, dtype=np.int64))
    order = np.lexsort((np.asarray(block_ids), -np.asarray(scores, dtype=F64)))
    return np.sort(np.asarray(block_ids, dtype=np.int64)[order[:k]])


# ---------------------------------------------------------------------------
# steps a4 / a5 / a6: attention and the exact log-sum-exp merge (fp64)
# ---------------------------------------------------------------------------

def attend(q: np.ndarray, kseq: np.ndarray, vseq: np.ndarray, tokens: np.ndarray, scale: float):
    """Softmax attention of one query over the given token positions, fp64.

    Returns (O [D], lse) with lse = log sum_t exp(z_t), z_t = scale * q.k_t
    (natural log).  An empty set gives (0, -inf)."""
    D = kseq.shape[1]
    if len(tokens) == 0:
        return np.zeros(D, dtype=F64), -math.inf
    K = kseq[tokens].astype(F64)
    V = vseq[tokens].astype(F64)
    z = scale * (K * np.asarray(q, dtype=F64)[None, :]).sum(axis=1)
    m = z.max()
    w = np.exp(z - m)
    s = w.sum()
    O = (w[:, None] * V).sum(axis=0) / s
    return O, m + math.log(s)


def attention_logits(q: np.ndarray, kseq: np.ndarray, tokens: np.ndarray, scale: float) -> np.ndarray:
    K = kseq[tokens].astype(F64)
    return scale * (K * np.asarray(q, dtype=F64)[None, :]).sum(axis=1)


def lse_merge(O_a, lse_a, O_b, lse_b):
    """HGCA log-sum-exp fusion of two partial attentions over disjoint sets,
    stabilised by the larger lse (review, minor comment on Sec. 3.3).
    Works row-wise on arrays: O [..., D], lse [...]."""
    O_a = np.asarray(O_a, dtype=F64)
    O_b = np.asarray(O_b, dtype=F64)
    lse_a = np.asarray(lse_a, dtype=F64)
    lse_b = np.asarray(lse_b, dtype=F64)
    m = np.maximum(lse_a, lse_b)
    both_empty = np.isneginf(m)
    m_safe = np.where(both_empty, 0.0, m)
    wa = np.where(np.isneginf(lse_a), 0.0, np.exp(lse_a - m_safe))
    wb = np.where(np.isneginf(lse_b), 0.0, np.exp(lse_b - m_safe))
    den = wa + wb
    den_safe = np.where(both_empty, 1.0, den)
    O = (wa[..., None] * O_a + wb[..., None] * O_b) / den_safe[..., None]
    O = np.where(both_empty[..., None], 0.0, O)
    lse = np.where(both_empty, -np.inf, m_safe + np.log(den_safe))
    return O, lse


# ---------------------------------------------------------------------------
# one decode step, composed (used by the parity tests)
# ---------------------------------------------------------------------------

def to_np(t) -> np.ndarray:
    """bf16 / int torch tensor -> numpy (float32 for floats: exact for bf16)."""
    import torch
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32):
        return t.detach().to("cpu").float().numpy()
    return t.detach().to("cpu").numpy()


def select_head(q32, kseq, L, S, W, Bs, k, mode):
    """Summaries -> canonical scores -> top-k for one query head.
    Returns (selected block ids ascending, candidate ids, scores)."""
    j0, j1 = candidate_blocks(L, S, W, Bs)
    ids = np.arange(j0, j1, dtype=np.int64)
    if j1 <= j0:
        return np.zeros(0, dtype=np.int64), ids, np.zeros(0, dtype=F32)
    if k >= j1 - j0:
        return ids.copy(), ids, None
    summ = summarize_sequence(kseq, Bs, mode, j0, j1)
    sc = score_blocks(q32, summ, mode)
    return topk_blocks(sc, ids, k), ids, sc


def decode_head(q32, kseq, vseq, L, S, W, Bs, sel_blocks, scale):
    """Dense partial over I, sparse partial over J, and their merge, fp64."""
    I = dense_tokens(L, S, W)
    J = sparse_tokens(L, S, W, Bs, sel_blocks)
    O_I, lse_I = attend(q32, kseq, vseq, I, scale)
    O_J, lse_J = attend(q32, kseq, vseq, J, scale)
    O, lse = lse_merge(O_I, lse_I, O_J, lse_J)
    return dict(O=O, lse=float(lse), O_I=O_I, lse_I=lse_I, O_J=O_J, lse_J=lse_J, I=I, J=J)


# ---------------------------------------------------------------------------
# step a7: vertical / slash score tables (reading R6)
# ---------------------------------------------------------------------------
#
# LFPS ("What carries the argument", Eq. (10)): per head, a table indexed by
# absolute key position (vertical) and one indexed by offset from the newest
# token (slash), both decayed by r = 0.95 every step and fed with the step's
# attention weights; HGCA's moving average of attention weights is the
# vertical table.  LFPS Eq. (9): candidates are expanded by offsets
# {-1, 0, 1, 2}.  HGCA: an entry is kept when its average exceeds
# beta / (number of densely attended entries).

DECAY = 0.95
EXPANSION_OFFSETS = (-1, 0, 1, 2)


def merged_weights(q, kseq, L: int, S: int, W: int, cand_tokens, scale: float):
    """Attended positions (I plus the candidate tokens inside M, ascending)
    and their merged softmax weights a_i = exp(z_i - lse), fp64."""
    s_end, w_beg = partition(L, S, W)
    J = sorted(set(int(t) for t in cand_tokens if s_end <= t < w_beg))
    pos = np.array(sorted(set(dense_tokens(L, S, W).tolist()) | set(J)), dtype=np.int64)
    if len(pos) == 0:
        return pos, np.zeros(0)
    z = attention_logits(q, kseq, pos, scale)
    m = z.max()
    lse = m + math.log(np.exp(z - m).sum())
    return pos, np.exp(z - lse)


def table_update(vert, slash, L_prev: int, att_pos, att_w, r: float = DECAY):
    """One decay-and-add step, fp64: T <- r T + (1 - r) a, with a the weight
    of the entry at the step of length L_prev (0 where not attended).
    Vertical entry i holds position i; slash entry d holds position
    L_prev - 1 - d."""
    n = len(vert)
    a_pos = np.zeros(n)
    att_pos = np.asarray(att_pos, dtype=np.int64)
    a_pos[att_pos] = att_w
    v_new = r * np.asarray(vert, dtype=F64) + (1.0 - r) * a_pos
    d = np.arange(n)
    src = L_prev - 1 - d
    a_sl = np.where((src >= 0) & (src < n), a_pos[np.clip(src, 0, n - 1)], 0.0)
    s_new = r * np.asarray(slash, dtype=F64) + (1.0 - r) * a_sl
    return v_new, s_new


def table_candidates(vert32, slash32, L: int, S: int, W: int, beta: float, kcap: int):
    """Candidate tokens for a step of length L from fp32 tables: seeds i in M
    with vert[i] > tau or slash[L - 1 - i] > tau (tau = fp32(beta) / fp32(|I|),
    compared in fp32), expanded by {-1, 0, 1, 2} and clipped to M; ascending.
    Returns (positions, overflowed): at most kcap, lowest positions kept."""
    vert32 = np.asarray(vert32, dtype=F32)
    slash32 = np.asarray(slash32, dtype=F32)
    s_end, w_beg = partition(L, S, W)
    n_dense = s_end + (L - w_beg)
    if w_beg <= s_end or n_dense == 0:
        return np.zeros(0, dtype=np.int64), False
    tau = F32(beta) / F32(n_dense)
    i = np.arange(s_end, w_beg)
    seed = (vert32[i] > tau) | (slash32[L - 1 - i] > tau)
    seeds = i[seed]
    cand = set()
    for o in EXPANSION_OFFSETS:
        for j in (seeds + o).tolist():
            if s_end <= j < w_beg:
                cand.add(j)
    out = np.array(sorted(cand), dtype=np.int64)
    return out[:kcap], len(out) > kcap


# ---------------------------------------------------------------------------
# variant: one selection shared by the query heads of a KV group (reading R9)
# ---------------------------------------------------------------------------

def group_scores(per_head_scores) -> np.ndarray:
    """Fp32 sum of the group's canonical block scores in head order, one
    rounding per addition (reading R9)."""
    acc = np.asarray(per_head_scores[0], dtype=F32).copy()
    for sc in per_head_scores[1:]:
        acc = (acc + np.asarray(sc, dtype=F32)).astype(F32)
    return acc


def select_group(q32_group, kseq, L, S, W, Bs, k, mode):
    """One block selection for all query heads of a KV head (reading R9):
    summaries -> each head's canonical scores -> their fp32 sum -> top-k.
    Returns (selected block ids ascending, candidate ids, group scores)."""
    j0, j1 = candidate_blocks(L, S, W, Bs)
    ids = np.arange(j0, j1, dtype=np.int64)
    if j1 <= j0:
        return np.zeros(0, dtype=np.int64), ids, np.zeros(0, dtype=F32)
    if k >= j1 - j0:
        return ids.copy(), ids, None
    summ = summarize_sequence(kseq, Bs, mode, j0, j1)
    sc = group_scores([score_blocks(q, summ, mode) for q in q32_group])
    return topk_blocks(sc, ids, k), ids, sc


# ---------------------------------------------------------------------------
# exact top-k inside the table candidates (reading R10)
# ---------------------------------------------------------------------------

def exact_token_topk(q32, kseq, cand_tokens, k: int):
    """Keep the k candidate tokens with the largest exact score q . k_t
    (canonical fp32 order of reading R4 with the key row as operand), ties to
    the lower position; ascending.  Returns (kept positions, scores of all
    candidates in list order)."""
    cand = np.asarray(cand_tokens, dtype=np.int64)
    if len(cand) == 0:
        return cand, np.zeros(0, dtype=F32)
    sc = canonical_dot(np.asarray(q32, dtype=F32), np.asarray(kseq, dtype=F32)[cand])
    return topk_blocks(sc, cand, k), sc


# ---------------------------------------------------------------------------
# variant: head-sparsity estimate and mean-value bypass (reading R11)
# ---------------------------------------------------------------------------

# LFPS, "Assumptions & free parameters": sparsity threshold epsilon = 0.85 and
# a local window of six recent tokens in Eq. (5).
BYPASS_EPS = 0.85
LOCAL_WINDOW = 6


def sparsity_partition(L: int):
    """Token classes of the estimate (reading R11): the sink token 0, the
    local tokens [max(1, L - 6), L) and the n global tokens [1, max(1, L - 6)).
    Returns (local positions, global positions)."""
    if L <= 0:
        return np.zeros(0, dtype=np.int64), np.zeros(0, dtype=np.int64)
    lo = max(1, L - LOCAL_WINDOW)
    return np.arange(lo, L, dtype=np.int64), np.arange(1, lo, dtype=np.int64)


def head_sparsity(q, kseq, L: int, scale: float):
    """LFPS's sink-proportion estimate for one query head (Eq. (5), Eq. (6),
    App. B.1 as read in R11), fp64.

    z_t = scale * q . k_t.  Sink mass e^{z_0}; local mass the sum of e^{z_t}
    over the local tokens; global mass n * exp(scale q . Kbar + scale^2 |q|^2
    sigma^2 / 2), the mean of e^z under independent normal key components
    with the global tokens' mean Kbar and mean per-dimension population
    variance sigma^2.  Returns (rho, lse_est): the sink's share of the three
    masses and the log of their sum.  L = 0 gives (0, -inf)."""
    if L <= 0:
        return 0.0, -math.inf
    q = np.asarray(q, dtype=F64)
    K = np.asarray(kseq[:L], dtype=F64)
    loc, glo = sparsity_partition(L)
    logs = [scale * float(K[0] @ q)]                      # the sink
    logs += [scale * float(K[t] @ q) for t in loc]
    n = len(glo)
    if n > 0:
        Kg = K[glo]
        kbar = Kg.mean(axis=0)
        var = ((Kg - kbar[None, :]) ** 2).mean(axis=0).mean()
        logs.append(math.log(n) + scale * float(kbar @ q) + 0.5 * scale * scale * float(q @ q) * var)
    m = max(logs)
    tot = sum(math.exp(x - m) for x in logs)
    return math.exp(logs[0] - m) / tot, m + math.log(tot)


def bypass_output(vseq, L: int) -> np.ndarray:
    """Output of a bypassed head (LFPS Algorithm 1, step 1): the mean value
    row over the L tokens, fp64.  L = 0 gives zeros."""
    D = vseq.shape[1]
    if L <= 0:
        return np.zeros(D, dtype=F64)
    return np.asarray(vseq[:L], dtype=F64).mean(axis=0)


def is_bypassed(rho: float, eps: float = BYPASS_EPS) -> bool:
    """A head is bypassed when its sink share exceeds epsilon (strict)."""
    return rho > eps
