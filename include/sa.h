/*
 * sa.h -- C ABI of libsa: decode-phase hybrid sparse attention over a paged
 * bf16 KV cache, hand-written CUDA for sm_103a (GB300).
 *
 * What the library computes, and where the pages define it:
 *   - Dense attention over the attention sinks and the recent window, sparse
 *     attention over selected older entries, merged exactly by the
 *     log-sum-exp identity  O = (e^lse_I O_I + e^lse_J O_J)/(e^lse_I + e^lse_J),
 *     lse_S = log sum_{j in S} e^{s_j}.
 *     ("HGCA: Hybrid GPU-CPU Attention for Long Context LLM Inference", review
 *     section "What carries the argument"; minor comment on Sec. 3.3.)
 *   - Per-head top-k selection of fixed-size KV blocks under a head-specific
 *     block size and budget.  ("An Efficient Hybrid Sparse Attention with
 *     CPU-GPU Parallelism for Long-Context Inference" (Fluxion), core claim,
 *     Fig. 2, Fig. 5.)
 *   - KV kept in fixed-size pages reached through a page table.  ("Unifying
 *     Sparse Attention with Hierarchical Memory for Scalable Long-Context LLM
 *     Serving", abstract and Fig. 6.)
 *   - Vertical / slash score tables with decay 0.95 and positional expansion
 *     by offsets {-1,0,1,2}.  ("Learn from the Past: Fast Sparse Indexing for
 *     Large Language Model Decoding", "What carries the argument", Eq. (9),
 *     Eq. (10).)
 *
 * Conventions shared by every call:
 *   - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *     never allocates or frees them.  `stream` is a cudaStream_t passed as
 *     void* (NULL = legacy default stream).  Calls are asynchronous on it.
 *   - Dtypes are fixed: Q, K, V and block summaries bf16 (passed as void*);
 *     scores, outputs, lse, logits and score tables fp32; indices, page tables,
 *     lengths and counts int32.  All tensors are dense, row-major, no padding.
 *   - Notation: B sequences, Hq query heads, Hk KV heads, G = Hq / Hk query
 *     heads per KV head (query head h uses KV head h / G), D = 128, P = page
 *     size (16), L = seq_lens[b] tokens in the cache INCLUDING the current
 *     token (L must not exceed max_pages_per_seq * P), S sinks, W window,
 *     Bs = block size of a KV head.
 *     Dense set I = [0, min(S,L)) U [max(L-W, min(S,L)), L); middle region M
 *     = the tokens between.  Candidate blocks are the blocks that meet M:
 *     j in [min(S,L)/Bs, ceil(max(L-W, min(S,L))/Bs)).  A selected block
 *     contributes only its tokens inside M, so I and the sparse set are
 *     disjoint.
 *   - KV pool layout: [num_pages][Hk][P][D] bf16 (one page of one KV head is a
 *     contiguous P x D slab).  Page table: [B][max_pages_per_seq] int32,
 *     logical page -> physical page.  Token t of sequence b is row t % P of
 *     physical page page_table[b][t / P].
 *   - Return value: SA_OK or an SA_ERR_* code.  Errors a host can see (bad
 *     arguments, unsupported shapes, capacity) return BEFORE any launch.
 *     Errors only the device can see (a page-table entry outside
 *     [0, num_pages), a bounded wait that ran out) set a status word in the
 *     workspace; the offending work is skipped, nothing traps.  Read it with
 *     sa_get_status().
 *   - Scratch comes from a caller-allocated workspace of sa_workspace_size()
 *     bytes (16-byte aligned), zeroed once with sa_workspace_init().  Calls
 *     that share one workspace must be ordered on one stream.
 *   - Alignment: q, the K / V pools, summaries, out and the workspace must be
 *     16-byte aligned (the kernels move them 16 bytes at a time); a
 *     misaligned pointer returns SA_ERR_INVALID_ARG before any launch.
 */
#ifndef SA_H_
#define SA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SA_OK 0
#define SA_ERR_INVALID_ARG 1
#define SA_ERR_UNSUPPORTED 2
#define SA_ERR_CUDA 3
#define SA_ERR_CAPACITY 4
#define SA_ERR_BAD_PAGE 5
#define SA_ERR_TIMEOUT 6

/* block summary kinds */
#define SA_SUMMARY_MINMAX 0 /* [..][2][D]: row 0 = per-dim min, row 1 = per-dim max */
#define SA_SUMMARY_MEAN 1   /* [..][D]: bf16(RNE(fp32 ascending sum / n)) */

/* how blocks are selected (sa_problem.selection_mode) */
#define SA_SELECT_PER_HEAD 0 /* each query head keeps its own top-k blocks */
#define SA_SELECT_GROUP 1    /* the G query heads of a KV head share one top-k, ranked by the fp32 sum
                                of their scores in head order; every head of a group must have the
                                same k.  A variant: the pages select per head. */

/* granularity of a selection list handed to sa_sparse_decode */
#define SA_SEL_BLOCK 0 /* entries are block indices of the head's KV head */
#define SA_SEL_TOKEN 1 /* entries are token positions */

/* sa_block_summarize: block_begin value meaning "only the block holding the
 * newest token L-1" (the incremental per-step refresh) */
#define SA_BLOCKS_TAIL (-1)

/* limits of this build */
#define SA_HEAD_DIM 128
#define SA_PAGE_SIZE 16
#define SA_MAX_GROUP 8   /* G <= 8 */
#define SA_MAX_HK 64
#define SA_MAX_HQ 256

/* Shapes and selection settings of one attention layer.  Host memory. */
typedef struct sa_problem {
  int32_t B;                   /* sequences */
  int32_t Hq;                  /* query heads */
  int32_t Hk;                  /* KV heads; Hq % Hk == 0, Hq / Hk <= 8 */
  int32_t D;                   /* head dim; must be 128 */
  int32_t page_size;           /* must be 16 */
  int32_t max_pages_per_seq;   /* columns of the page table */
  int32_t num_pages;           /* physical pages in each pool */
  int32_t sink;                /* S >= 0 */
  int32_t window;              /* W >= max block size */
  int32_t summary_mode;        /* SA_SUMMARY_MINMAX or SA_SUMMARY_MEAN */
  const int32_t* block_size_per_kvh; /* host [Hk], each in {8,16,32,64} */
  const int32_t* k_per_qhead;        /* host [Hq], blocks kept per head, 0 <= k <= kcap */
  int32_t kcap;                /* capacity of a selection list (entries per head) */
  float scale;                 /* softmax scale, normally 1/sqrt(D) */
  int32_t selection_mode;      /* SA_SELECT_PER_HEAD (0, the pages' selection) or SA_SELECT_GROUP */
} sa_problem;

/* Block slots per (sequence, KV head) in the summary and score tensors:
 * ceil(max_pages_per_seq * page_size / min block size).  Block j of KV head
 * kvh of sequence b lives at slot [b][kvh][j].  0 if prob is invalid. */
int32_t sa_block_slots(const sa_problem* prob);

/* Workspace bytes for calls on this problem (0 if prob is invalid). */
size_t sa_workspace_size(const sa_problem* prob);

/* Zero a workspace (async on stream).  Needed once before first use and after
 * any call that reported SA_ERR_TIMEOUT. */
int sa_workspace_init(void* ws, size_t bytes, void* stream);

/* Synchronise `stream`, read the device status word of `ws` into *status
 * (SA_OK if no device-side error since the last read) and clear it. */
int sa_get_status(void* ws, void* stream, int* status);

/* Human-readable message for a status code (static storage). */
const char* sa_status_string(int status);

/* Step a1 -- block summaries.
 * For every (b, kvh) and block j in [block_begin, block_end) clipped to
 * [0, ceil(L/Bs)), summarise tokens [j Bs, min((j+1) Bs, L)) of K:
 * MINMAX writes summaries[b][kvh][j][0][:] = min, [1][:] = max (exact);
 * MEAN writes summaries[b][kvh][j][:] = bf16(RNE(fp32 sum in ascending token
 * order / n)).  block_end = -1 means through the last block; block_begin =
 * SA_BLOCKS_TAIL means only the block holding token L-1 (per-step refresh).
 * Layout: [B][Hk][sa_block_slots][2][D] (MINMAX) or [B][Hk][slots][D] (MEAN),
 * bf16.  The pages do not define the summary; this is the min/max bounding
 * box or the mean key (Fluxion core claim: block-level selection).
 * Device errors: a bad page id sets SA_ERR_BAD_PAGE, the block is written 0. */
int sa_block_summarize(const sa_problem* prob, const void* k_pool,
                       const int32_t* page_table, const int32_t* seq_lens,
                       int32_t block_begin, int32_t block_end, void* summaries,
                       void* ws, void* stream);

/* Step a2 -- block scores.  Fluxion (core claim; Fig. 2d, where the top-k
 * cost grows as blocks shrink) ranks KV blocks per head, and LFPS ("The
 * reading") notes that an exact top-k needs a dot product against every
 * key; the pages do not define the block score itself.  The score taken
 * here is the dot product of q with the block summary of sa_block_summarize:
 * for every (b, query head h) and candidate block j,
 * MINMAX  s = sum_d q_d * (q_d >= 0 ? kmax_d : kmin_d)  (the largest q.k any
 *         key inside the block's min/max box can reach)
 * MEAN    s = sum_d q_d * kmean_d
 * in fp32 in the canonical order: the 128 dims form 8 lanes of 16
 * consecutive dims, each lane sums its exact products in ascending dim order
 * (one rounding per step), the 8 lane sums are combined by a butterfly with
 * partner offsets 4, 2, 1, and +0.0 is added.  Unscaled.
 * scores: [B][Hq][sa_block_slots] fp32; only candidate slots are written. */
int sa_score_blocks(const sa_problem* prob, const void* q,
                    const void* summaries, const int32_t* seq_lens,
                    float* scores, void* ws, void* stream);

/* Steps a2 + a3 -- fused score and per-head top-k.  For every (b, h): keep
 * k_h = min(k_per_qhead[h], ncand) candidate blocks, ranked by score
 * descending then block index ascending, written ascending to
 * sel_idx[b][h][0..k_h) with sel_cnt[b][h] = k_h.  If k_h == ncand the head
 * keeps every candidate without scoring (a 100 % budget is dense attention).
 * sel_idx: [B][Hq][kcap] int32; sel_cnt: [B][Hq] int32.
 * scores_or_null: if not NULL, the scores are also written as in
 * sa_score_blocks.  Requires k_per_qhead[h] <= kcap (else SA_ERR_CAPACITY).
 * With prob->selection_mode == SA_SELECT_GROUP the ranking of a KV head's
 * blocks is the fp32 sum of its G heads' scores, added in head order, and the
 * G rows of sel_idx / sel_cnt receive the same list (a variant: Fluxion's
 * core claim selects per head). */
int sa_select_topk(const sa_problem* prob, const void* q,
                   const void* summaries, const int32_t* seq_lens,
                   int32_t* sel_idx, int32_t* sel_cnt, float* scores_or_null,
                   void* ws, void* stream);

/* Steps a4 + a5 + a6 -- paged gather split-K decode attention with the exact
 * log-sum-exp merge.  HGCA (review, "What carries the argument") attends the
 * newest entries densely and selected older entries sparsely and fuses the
 * two partial outputs with the identity above; SPIN (abstract, Fig. 6) keeps
 * the KV in pages reached through a page table; Fluxion (Fig. 4) keeps the
 * attention sinks.  For every (b, h): attend q[b][h] over I plus the
 * head's selected set J_h = (entries of sel_idx[b][h][0..sel_cnt)) inside M,
 * with z_t = scale * q.k_t:
 *   out[b][h][:] = sum_t softmax(z)_t v_t  (fp32), lse[b][h] = log sum e^{z_t}.
 * Entries outside M or beyond L are ignored; duplicates count once.  The KV
 * rows of the union over a KV head's G query heads are read once.  Work is
 * split into chunks of pages whose partials (max, sum, O) are combined with
 * the identity above, in chunk order, by a second kernel on the same stream
 * (no host synchronisation).  An empty attended set (L = 0)
 * gives out = 0, lse = -inf.
 * sel_granularity: SA_SEL_BLOCK (entries are blocks of the KV head's Bs) or
 *   SA_SEL_TOKEN (entries are positions).
 * logits_or_null: if not NULL, [B][Hq][max_pages_per_seq*P] fp32 receives the
 *   natural-log-domain logit z_t at every attended position t (other positions
 *   untouched).  Used to feed the score-table update.
 * bypass_or_null: if not NULL, [B][Hq] int32 as sa_head_sparsity writes it:
 *   a head with a non-zero entry is left out (its selection ignored, no KV
 *   read for it alone) and its out / lse rows are not written.
 * out: [B][Hq][D] fp32; lse: [B][Hq] fp32 (natural log). */
int sa_sparse_decode(const sa_problem* prob, const void* q,
                     const void* k_pool, const void* v_pool,
                     const int32_t* page_table, const int32_t* seq_lens,
                     const int32_t* sel_idx, const int32_t* sel_cnt,
                     int32_t sel_granularity, float* out, float* lse,
                     float* logits_or_null, const int32_t* bypass_or_null,
                     void* ws, void* stream);

/* One whole decode step for block selection -- a1 (incremental) + a2 + a3 +
 * a4 + a5 + a6: the same results as
 *   sa_block_summarize(prob, k_pool, page_table, seq_lens, SA_BLOCKS_TAIL, -1,
 *                      summaries, ws, stream);
 *   sa_select_topk(prob, q, summaries, seq_lens, sel_idx, sel_cnt, NULL, ws, stream);
 *   sa_sparse_decode(prob, q, k_pool, v_pool, page_table, seq_lens, sel_idx,
 *                    sel_cnt, SA_SEL_BLOCK, out, lse, NULL, ws, stream);
 * in fewer launches (the tile list and the tail-block summary share one
 * kernel per KV head).  summaries are read for scoring and their tail
 * block rewritten; sel_idx / sel_cnt receive the selection. */
int sa_decode_step(const sa_problem* prob, const void* q, const void* k_pool,
                   const void* v_pool, const int32_t* page_table,
                   const int32_t* seq_lens, void* summaries, int32_t* sel_idx,
                   int32_t* sel_cnt, float* out, float* lse, void* ws,
                   void* stream);

/* A prepared decode step: sa_decode_step on fixed buffers, captured once into
 * a CUDA graph inside the library and replayed by one call.  For a serving
 * loop that reuses its buffers (fresh contents each step, same addresses):
 * the launch costs one graph launch on the host instead of the step's
 * argument checks, descriptor set-up and four kernel launches.
 *   sa_step_plan_create: checks the arguments as sa_decode_step does (the
 *     same errors, returned before anything is captured), then captures the
 *     step's launches on a private stream and instantiates the graph.  Not
 *     inside a stream capture.  Allocates host and graph resources.
 *   sa_step_plan_launch: one sa_decode_step on the plan's buffers, async on
 *     `stream`; the buffers' current contents are used.  Calls that share the
 *     plan's workspace must be ordered on one stream.
 *   sa_step_plan_destroy: frees the plan (NULL is a no-op); the caller keeps
 *     the buffers. */
typedef struct sa_step_plan sa_step_plan;

int sa_step_plan_create(const sa_problem* prob, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* page_table, const int32_t* seq_lens, void* summaries, int32_t* sel_idx,
                        int32_t* sel_cnt, float* out, float* lse, void* ws, sa_step_plan** plan);
int sa_step_plan_launch(sa_step_plan* plan, void* stream);
int sa_step_plan_destroy(sa_step_plan* plan);

/* The new token's key and value rows into the pools: for every (b, kv head)
 * with L = seq_lens[b] > 0 (L counts the new token), k_new[b][kvh][:] and
 * v_new[b][kvh][:] (bf16 [B][Hk][D], 16-byte aligned) are written at
 * position L - 1, i.e. row (L - 1) % P of page page_table[b][(L - 1) / P].
 * A page outside the pool records SA_ERR_BAD_PAGE and writes nothing.
 * (SPIN, abstract and Fig. 6: the paged KV substrate.) */
int sa_append_kv(const sa_problem* prob, const void* k_new, const void* v_new,
                 void* k_pool, void* v_pool, const int32_t* page_table,
                 const int32_t* seq_lens, void* ws, void* stream);

/* sa_decode_step preceded by the append of the new token: the same results as
 *   sa_append_kv(prob, k_new, v_new, k_pool, v_pool, page_table, seq_lens, ws, stream);
 *   sa_decode_step(prob, q, k_pool, v_pool, page_table, seq_lens, summaries,
 *                  sel_idx, sel_cnt, out, lse, ws, stream);
 * with the append done inside the step (by the warp that refreshes the tail
 * summary, after the scores, which never read the newest token's block). */
int sa_decode_step_append(const sa_problem* prob, const void* q,
                          const void* k_new, const void* v_new, void* k_pool,
                          void* v_pool, const int32_t* page_table,
                          const int32_t* seq_lens, void* summaries,
                          int32_t* sel_idx, int32_t* sel_cnt, float* out,
                          float* lse, void* ws, void* stream);

/* Step a7 -- score-table update and table-driven candidate selection.
 * Tables: vertical (entry i = absolute position i) and slash (entry d =
 * offset d from the newest token, i.e. position L - 1 - d), fp32
 * [B][Hq][max_pages_per_seq * P], one row per query head.  They are
 * double-buffered: *_in is read, *_out written; out must not overlap in.
 * Update (when prev_logits != NULL): with the previous decode step of length
 * Lp = prev_seq_lens[b] (attended set = its dense set plus the sorted token
 * list prev_sel_idx[b][h][0..prev_sel_cnt) inside its middle region, logits
 * and lse as written by sa_sparse_decode), every entry becomes
 *   T_out = fma(decay, T_in, (1 - decay) * exp(z - lse))   (attended)
 *   T_out = decay * T_in                                 (not attended)
 * in fp32; the slash entry d takes the weight of position Lp - 1 - d.
 * Without prev_logits the tables are copied unchanged; so are the rows of
 * heads with a non-zero prev_bypass_or_null[b][h] ([B][Hq] int32, the
 * previous step's sa_head_sparsity flags: LFPS leaves a bypassed head's
 * tables as they were).
 * Selection for the next step of length L = seq_lens[b]: position i in the
 * middle region M of L is a seed if vert_out[i] > tau or slash_out[L-1-i] >
 * tau, tau = beta / |I(L)| (fp32, strict); candidates are the seeds expanded
 * by offsets {-1, 0, 1, 2} and clipped to M, written ascending to
 * cand_idx[b][h][0..kcap) with cand_cnt[b][h]; beyond kcap the lowest are
 * kept and SA_ERR_CAPACITY is recorded in the workspace status word.
 * (LFPS: "What carries the argument", Eq. (9), Eq. (10), r = 0.95; HGCA:
 * moving average of attention weights and its beta / N threshold.) */
int sa_update_score_tables(const sa_problem* prob, const float* vert_in,
                           const float* slash_in, float* vert_out,
                           float* slash_out, const int32_t* prev_seq_lens,
                           const int32_t* prev_sel_idx,
                           const int32_t* prev_sel_cnt,
                           const float* prev_logits, const float* prev_lse,
                           const int32_t* prev_bypass_or_null,
                           const int32_t* seq_lens, float decay, float beta,
                           int32_t* cand_idx, int32_t* cand_cnt, void* ws,
                           void* stream);

/* Sparse decode without a workspace.  The pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory and so
 * cannot hand sa_sparse_decode a workspace -- for example code running inside
 * a host framework that owns every device allocation through its own pool,
 * or a latency-critical path where cudaMalloc's implicit synchronisation is
 * not allowed.  The inputs, outputs and results of sa_sparse_decode with
 * bypass_or_null = NULL: there is no bypass input, every head attends.  The
 * scratch lives in a fixed 64 MiB array of device memory inside the library
 * (held by every GPU that loads the library until the process exits).
 * The call allocates nothing.  A problem whose scratch does not fit returns
 * SA_ERR_CAPACITY before any launch.
 * status_or_null: optional device int32 that receives the first device-side
 *   error of this call (SA_OK otherwise); it is zeroed at the start of the
 *   call.  When NULL, device-side errors are recorded only inside the library.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, and again after the
 * device's context changes (cudaDeviceReset); make that first call before
 * any stream capture.  All calls share the array and it keeps the last
 * call's contents (the status word is cleared at the start of each call and
 * the chunk ticket by the call's first kernel): calls that overlap on the
 * GPU race with each other. */
int sa_sparse_decode_noalloc(const sa_problem* prob, const void* q,
                             const void* k_pool, const void* v_pool,
                             const int32_t* page_table, const int32_t* seq_lens,
                             const int32_t* sel_idx, const int32_t* sel_cnt,
                             int32_t sel_granularity, float* out, float* lse,
                             float* logits_or_null, int32_t* status_or_null,
                             void* stream);

/* Exact top-k inside the score-table candidates (LFPS, "The reading": an
 * exact top-k needs a dot product against every key, the tables narrow the
 * keys down).  For every (b, h): the candidates cand_idx[b][h][0..cand_cnt)
 * (token positions, as sa_update_score_tables writes them) are scored by
 * q[b][h] . k_t in the canonical fp32 order of sa_score_blocks with the bf16
 * key row as operand; the k_per_qhead[h] best by (score descending, position
 * ascending) are written ascending to sel_idx[b][h] (sa_sparse_decode with
 * SA_SEL_TOKEN takes them) and their count to sel_cnt[b][h].  Entries outside
 * [0, L) rank last.
 * cand_idx, sel_idx: [B][Hq][kcap] int32; cand_cnt, sel_cnt: [B][Hq] int32.
 * scores_or_null: if not NULL, [B][Hq][kcap] fp32 receives the score of every
 * candidate at its list index.  kcap above 25600 gives SA_ERR_UNSUPPORTED. */
int sa_select_tokens(const sa_problem* prob, const void* q, const void* k_pool,
                     const int32_t* page_table, const int32_t* seq_lens,
                     const int32_t* cand_idx, const int32_t* cand_cnt,
                     int32_t* sel_idx, int32_t* sel_cnt, float* scores_or_null,
                     void* ws, void* stream);

/* Head-sparsity bypass (LFPS, "Learn from the Past": Algorithm 1 step 1,
 * Eq. (5), Eq. (6), App. B.1, epsilon = 0.85).  A variant, off unless these
 * calls are made.
 *
 * kv_stats: [B][Hk][3][D] fp32, per (b, kv head) the sums over the L =
 * seq_lens[b] cached tokens of k, of k*k (per dimension) and of v; 16-byte
 * aligned.  sa_kv_stats computes them from the cache in one pass (sums in
 * fp32, in a fixed order); sa_decode_step_bypass with k_new keeps them
 * current as tokens are appended.
 *
 * sa_head_sparsity: for every (b, h) with logits z_t = scale q . k_t, the
 * sink token 0, the local window [max(1, L - 6), L) and the n = max(0, L - 7)
 * global tokens between:
 *   m_sink = e^{z_0}, m_local = sum over the window of e^{z_t},
 *   m_global = n exp(scale q . Kbar + scale^2 |q|^2 sigma^2 / 2)
 * with Kbar the global keys' mean and sigma^2 the mean over dims of their
 * per-dim variance (from kv_stats minus the sink and window rows) -- the
 * log-normal mean of e^z.  rho = m_sink / (m_sink + m_local + m_global)
 * (fp32) goes to rho_or_null[b][h]; bypass[b][h] = rho > eps (0 <= eps <= 1,
 * else SA_ERR_INVALID_ARG).  For a bypassed head out[b][h][:] = sum v / L and
 * lse[b][h] = log(m_sink + m_local + m_global); other rows of out / lse are
 * not touched.  L = 0 is never bypassed.  A page outside the pool records
 * SA_ERR_BAD_PAGE and leaves the head unbypassed.
 * rho_or_null: [B][Hq] fp32; bypass: [B][Hq] int32; out: [B][Hq][D] fp32,
 * lse: [B][Hq] fp32 (16-byte aligned out). */
int sa_kv_stats(const sa_problem* prob, const void* k_pool, const void* v_pool,
                const int32_t* page_table, const int32_t* seq_lens,
                float* kv_stats, void* ws, void* stream);

int sa_head_sparsity(const sa_problem* prob, const void* q, const void* k_pool,
                     const int32_t* page_table, const int32_t* seq_lens,
                     const float* kv_stats, float eps, float* rho_or_null,
                     int32_t* bypass, float* out, float* lse, void* ws,
                     void* stream);

/* The decode step with the bypass: the same results as
 *   [sa_append_kv(...) and the new rows added to kv_stats, when k_new_or_null]
 *   sa_head_sparsity(prob, q, k_pool, page_table, seq_lens, kv_stats, eps,
 *                    rho_or_null, bypass, out, lse, ws, stream);
 *   sa_decode_step(...)   with the bypassed heads left out:
 * a bypassed head gets sel_cnt = 0, no KV is read for it alone, and its out /
 * lse rows keep the bypass output.  k_new_or_null and v_new_or_null are both
 * NULL or both set (bf16 [B][Hk][D]; then L = seq_lens[b] counts the new
 * token and kv_stats must cover the L - 1 tokens before it on entry). */
int sa_decode_step_bypass(const sa_problem* prob, const void* q,
                          const void* k_new_or_null, const void* v_new_or_null,
                          void* k_pool, void* v_pool,
                          const int32_t* page_table, const int32_t* seq_lens,
                          void* summaries, float* kv_stats, float eps,
                          int32_t* sel_idx, int32_t* sel_cnt, float* out,
                          float* lse, float* rho_or_null, int32_t* bypass,
                          void* ws, void* stream);

/* Step a6 standalone -- merge two partial attentions over disjoint sets:
 * m = max(lse_a, lse_b), w_x = e^{lse_x - m},
 * o = (w_a o_a + w_b o_b) / (w_a + w_b), lse = m + log(w_a + w_b);
 * a side with lse = -inf contributes nothing; both -inf gives o = 0,
 * lse = -inf.  o_*: [n_rows][D] fp32; lse_*: [n_rows] fp32.  Output may alias
 * an input.  (HGCA review, "What carries the argument" and Sec. 3.3.) */
int sa_lse_merge(int32_t n_rows, int32_t D, const float* o_a,
                 const float* lse_a, const float* o_b, const float* lse_b,
                 float* o, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SA_H_ */
