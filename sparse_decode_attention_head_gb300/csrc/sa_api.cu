// The C ABI of libsa (declared in include/sa.h): argument validation,
// workspace layout, TMA descriptors, and the launches.  Everything a host can
// check is checked here, before any launch.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "launch.cuh"


using sa::Params;

// Host-side helpers (also used by noalloc.cu).
namespace sa_host {

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Validate a problem and fill the launch parameters.
int make_params(const sa_problem* pr, Params* p) {
  if (pr == nullptr) return SA_ERR_INVALID_ARG;
  if (pr->B < 1 || pr->Hq < 1 || pr->Hk < 1) return SA_ERR_INVALID_ARG;
  if (pr->Hq % pr->Hk != 0) return SA_ERR_INVALID_ARG;
  if (pr->D != SA_HEAD_DIM) return SA_ERR_INVALID_ARG;
  if (pr->Hq / pr->Hk > SA_MAX_GROUP || pr->Hk > SA_MAX_HK || pr->Hq > SA_MAX_HQ) return SA_ERR_UNSUPPORTED;
  if (pr->page_size != SA_PAGE_SIZE) return SA_ERR_UNSUPPORTED;
  if (pr->max_pages_per_seq < 1 || pr->num_pages < 1 || pr->sink < 0) return SA_ERR_INVALID_ARG;
  if (pr->summary_mode != SA_SUMMARY_MINMAX && pr->summary_mode != SA_SUMMARY_MEAN) return SA_ERR_INVALID_ARG;
  if (pr->block_size_per_kvh == nullptr || pr->k_per_qhead == nullptr) return SA_ERR_INVALID_ARG;
  if (pr->kcap < 1) return SA_ERR_INVALID_ARG;
  if (pr->selection_mode != SA_SELECT_PER_HEAD && pr->selection_mode != SA_SELECT_GROUP) return SA_ERR_INVALID_ARG;
  if (!(pr->scale > 0.f) || !std::isfinite(pr->scale)) return SA_ERR_INVALID_ARG;
  if ((long long)pr->max_pages_per_seq * SA_PAGE_SIZE >= (1LL << 30)) return SA_ERR_UNSUPPORTED;
  if ((long long)pr->num_pages * pr->Hk * SA_PAGE_SIZE >= (1LL << 31)) return SA_ERR_UNSUPPORTED;
  int max_bs = 0, min_bs = 1 << 30;
  for (int i = 0; i < pr->Hk; ++i) {
    const int bs = pr->block_size_per_kvh[i];
    if (bs != 8 && bs != 16 && bs != 32 && bs != 64) return SA_ERR_INVALID_ARG;
    if (!(SA_PAGE_SIZE % bs == 0 || bs % SA_PAGE_SIZE == 0)) return SA_ERR_INVALID_ARG;
    max_bs = std::max(max_bs, bs);
    min_bs = std::min(min_bs, bs);
  }
  if (pr->window < max_bs) return SA_ERR_INVALID_ARG;   // every candidate block is then complete
  for (int i = 0; i < pr->Hq; ++i) {
    if (pr->k_per_qhead[i] < 0) return SA_ERR_INVALID_ARG;
    if (pr->k_per_qhead[i] > pr->kcap) return SA_ERR_CAPACITY;
    // a shared selection needs one budget per group
    if (pr->selection_mode == SA_SELECT_GROUP && pr->k_per_qhead[i] != pr->k_per_qhead[i - i % (pr->Hq / pr->Hk)])
      return SA_ERR_INVALID_ARG;
  }
  std::memset(p, 0, sizeof(*p));
  p->sel_mode = pr->selection_mode;
  p->B = pr->B;
  p->Hq = pr->Hq;
  p->Hk = pr->Hk;
  p->G = pr->Hq / pr->Hk;
  p->mpp = pr->max_pages_per_seq;
  p->num_pages = pr->num_pages;
  p->S = pr->sink;
  p->W = pr->window;
  p->mode = pr->summary_mode;
  p->kcap = pr->kcap;
  p->scale = pr->scale;
  p->slots = (int)(((long long)pr->max_pages_per_seq * SA_PAGE_SIZE + min_bs - 1) / min_bs);
  for (int i = 0; i < pr->Hk; ++i) p->bs[i] = pr->block_size_per_kvh[i];
  for (int i = 0; i < pr->Hq; ++i) p->k[i] = pr->k_per_qhead[i];
  return SA_OK;
}

struct Layout {
  size_t header, scores, tiles, ntiles, ticket, partials, stage, total;
};

Layout layout_of(const Params& p) {
  Layout l;
  size_t off = 0;
  l.header = off;
  off = align_up(off + sizeof(sa::WsHeader));
  l.scores = off;
  off = align_up(off + (size_t)p.B * p.Hq * p.slots * sizeof(float));
  l.tiles = off;
  off = align_up(off + sa::tiles_bytes(p));
  l.ntiles = off;   // tile counts per (unit, window)
  off = align_up(off + sa::ntiles_bytes(p));
  l.ticket = off;   // the decode's chunk ticket (zeroed by the tile builder)
  off = align_up(off + sizeof(int));
  l.partials = off;
  off = align_up(off + sa::decode_partials_bytes(p));
  l.stage = off;   // score-table candidates per chunk
  off = align_up(off + sa::tables_stage_bytes(p));
  l.total = off;
  return l;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Pool [num_pages][Hk][P][D] bf16 viewed as rows of D; boxes of 16 rows x 64.
int encode_kv_map(CUtensorMap* m, const void* pool, const Params& p);

// The last few maps a host thread encoded, keyed by pool address, shape and
// device: a decode step needs two, and encoding is host work worth skipping.
int make_kv_map(CUtensorMap* m, const void* pool, const Params& p) {
  struct Entry {
    const void* pool;
    int num_pages, Hk, dev;
    CUtensorMap map;
  };
  thread_local Entry cache[8] = {};
  thread_local int next = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  for (const Entry& e : cache)
    if (e.pool == pool && pool != nullptr && e.num_pages == p.num_pages && e.Hk == p.Hk && e.dev == dev) {
      *m = e.map;
      return SA_OK;
    }
  const int rc = encode_kv_map(m, pool, p);
  if (rc == SA_OK) {
    cache[next] = Entry{pool, p.num_pages, p.Hk, dev, *m};
    next = (next + 1) % 8;
  }
  return rc;
}

int encode_kv_map(CUtensorMap* m, const void* pool, const Params& p) {
  auto fn = encode_fn();
  if (fn == nullptr) return SA_ERR_CUDA;
  // the pool as (64 dims, rows, 2 halves of a row): one box of 64 x 16 x 2
  // is a whole 4 KB page slab, landing as [half][row][64] with the 128-byte
  // swizzle, the layout two 64 x 16 boxes of a 2-D map would give
  cuuint64_t dims[3] = {64, (cuuint64_t)p.num_pages * p.Hk * SA_PAGE_SIZE, 2};
  cuuint64_t strides[2] = {(cuuint64_t)SA_HEAD_DIM * 2, 128};
  cuuint32_t box[3] = {64, 16, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? SA_OK : SA_ERR_CUDA;
}

int num_sms_current() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev < 64) cache[dev] = n;
  return n;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }


}  // namespace sa_host

using namespace sa_host;

extern "C" {

int32_t sa_block_slots(const sa_problem* prob) {
  Params p;
  if (make_params(prob, &p) != SA_OK) return 0;
  return p.slots;
}

size_t sa_workspace_size(const sa_problem* prob) {
  Params p;
  if (make_params(prob, &p) != SA_OK) return 0;
  return layout_of(p).total;
}

int sa_workspace_init(void* ws, size_t bytes, void* stream) {
  if (ws == nullptr || bytes < sizeof(sa::WsHeader)) return SA_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, bytes, as_stream(stream)) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int sa_get_status(void* ws, void* stream, int* status) {
  if (ws == nullptr || status == nullptr) return SA_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SA_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(int), s) != cudaSuccess) return SA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SA_ERR_CUDA;
  *status = v;
  return SA_OK;
}

const char* sa_status_string(int status) {
  switch (status) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported shape or setting";
    case SA_ERR_CUDA: return "CUDA runtime error";
    case SA_ERR_CAPACITY: return "capacity exceeded";
    case SA_ERR_BAD_PAGE: return "page-table entry outside the pool";
    case SA_ERR_TIMEOUT: return "bounded device wait ran out";
    default: return "unknown status";
  }
}

int sa_block_summarize(const sa_problem* prob, const void* k_pool, const int32_t* page_table,
                       const int32_t* seq_lens, int32_t block_begin, int32_t block_end, void* summaries,
                       void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!k_pool || !page_table || !seq_lens || !summaries || !ws) return SA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(summaries) || !aligned16(ws)) return SA_ERR_INVALID_ARG;
  if (block_begin < 0 && block_begin != SA_BLOCKS_TAIL) return SA_ERR_INVALID_ARG;
  if (block_end < -1) return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  return sa::launch_summarize(p, k_pool, page_table, seq_lens, block_begin, block_end, summaries,
                              at<int>(ws, l.header), as_stream(stream));
}

int sa_score_blocks(const sa_problem* prob, const void* q, const void* summaries, const int32_t* seq_lens,
                    float* scores, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !summaries || !seq_lens || !scores || !ws) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summaries) || !aligned16(ws)) return SA_ERR_INVALID_ARG;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SA_ERR_CUDA;
  return sa::launch_score(p, q, summaries, seq_lens, scores, 1, nsm, as_stream(stream), nullptr);
}

int sa_select_topk(const sa_problem* prob, const void* q, const void* summaries, const int32_t* seq_lens,
                   int32_t* sel_idx, int32_t* sel_cnt, float* scores_or_null, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !summaries || !seq_lens || !sel_idx || !sel_cnt || !ws) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(summaries) || !aligned16(ws)) return SA_ERR_INVALID_ARG;
  if (sa::topk_smem_bytes(p) > 200 * 1024) return SA_ERR_UNSUPPORTED;
  const Layout l = layout_of(p);
  float* scores = scores_or_null ? scores_or_null : at<float>(ws, l.scores);
  cudaStream_t s = as_stream(stream);
  const int nsm = num_sms_current();
  if (nsm <= 0) return SA_ERR_CUDA;
  rc = sa::launch_score(p, q, summaries, seq_lens, scores, scores_or_null != nullptr, nsm, s, nullptr);
  if (rc != SA_OK) return rc;
  return sa::launch_topk(p, scores, seq_lens, sel_idx, sel_cnt, s);
}

int sa_sparse_decode(const sa_problem* prob, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* page_table, const int32_t* seq_lens, const int32_t* sel_idx,
                     const int32_t* sel_cnt, int32_t sel_granularity, float* out, float* lse,
                     float* logits_or_null, const int32_t* bypass_or_null, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  p.bypass = bypass_or_null;
  if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !sel_idx || !sel_cnt || !out || !lse || !ws)
    return SA_ERR_INVALID_ARG;
  if (sel_granularity != SA_SEL_BLOCK && sel_granularity != SA_SEL_TOKEN) return SA_ERR_INVALID_ARG;
  // the kernels read q, K, V with 16-byte copies and store out and the
  // workspace's tiles and partials 16 bytes at a time
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) || !aligned16(ws))
    return SA_ERR_INVALID_ARG;
  if ((size_t)p.mpp * sizeof(int) > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (sa::decode_smem_bytes(p) > 227 * 1024) return SA_ERR_UNSUPPORTED;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SA_ERR_CUDA;
  CUtensorMap tmK, tmV;
  if ((rc = make_kv_map(&tmK, k_pool, p)) != SA_OK) return rc;
  if ((rc = make_kv_map(&tmV, v_pool, p)) != SA_OK) return rc;
  const Layout l = layout_of(p);
  cudaStream_t s = as_stream(stream);
  rc = sa::launch_build_tiles(p, seq_lens, page_table, sel_idx, sel_cnt, sel_granularity, at<void>(ws, l.tiles),
                              at<int>(ws, l.ntiles), at<int>(ws, l.header),
                              at<int>(ws, l.ticket), s);
  if (rc != SA_OK) return rc;
  return sa::launch_decode(p, q, page_table, at<void>(ws, l.tiles), at<int>(ws, l.ntiles),
                           at<float>(ws, l.partials), at<int>(ws, l.ticket), out, lse, logits_or_null,
                           at<int>(ws, l.header), tmK, tmV, nsm, s);
}

}  // extern "C"

namespace sa_host {

// sa_decode_step, and with k_new / v_new the appending variant.
// With kv_stats the step starts with the sparsity estimate (which then also
// does the append) and leaves the bypassed heads out of everything after it.
int decode_step_impl(const sa_problem* prob, const void* q, const void* k_new, const void* v_new, const void* k_pool,
                     const void* v_pool, const int32_t* page_table, const int32_t* seq_lens, void* summaries,
                     int32_t* sel_idx, int32_t* sel_cnt, float* out, float* lse, void* ws, void* stream,
                     float* kv_stats = nullptr, float eps = 1.f, float* rho = nullptr, int32_t* bypass = nullptr) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (kv_stats != nullptr && (bypass == nullptr || !(eps >= 0.f && eps <= 1.f))) return SA_ERR_INVALID_ARG;
  if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !summaries || !sel_idx || !sel_cnt || !out || !lse ||
      !ws)
    return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(summaries) || !aligned16(out) ||
      !aligned16(ws))
    return SA_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return SA_ERR_INVALID_ARG;
  if (k_new != nullptr && (!aligned16(k_new) || !aligned16(v_new))) return SA_ERR_INVALID_ARG;
  if ((size_t)p.mpp * sizeof(int) > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (sa::decode_smem_bytes(p) > 227 * 1024) return SA_ERR_UNSUPPORTED;
  const int nsm = num_sms_current();
  if (nsm <= 0) return SA_ERR_CUDA;
  CUtensorMap tmK, tmV;
  if ((rc = make_kv_map(&tmK, k_pool, p)) != SA_OK) return rc;
  if ((rc = make_kv_map(&tmV, v_pool, p)) != SA_OK) return rc;
  const Layout l = layout_of(p);
  cudaStream_t s = as_stream(stream);
  int* status = at<int>(ws, l.header);
  float* scores = at<float>(ws, l.scores);
  void* kp = const_cast<void*>(k_pool);
  void* vp = const_cast<void*>(v_pool);
  // the head-sparsity estimate runs in the score kernel's first warps; it
  // takes the new token's rows from k_new / v_new (the append, and their
  // addition to the sums, follow in the tile-building kernel)
  sa::EstArgs E{};
  if (kv_stats != nullptr) {
    E = sa::EstArgs{static_cast<const __nv_bfloat16*>(k_pool), page_table,
                    static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), kv_stats,
                    eps, rho, bypass, out, lse, status};
  }
  // the scores never read the newest token's block (it is in the window), so
  // the append and the tail summary can follow them
  if ((rc = sa::launch_score(p, q, summaries, seq_lens, scores, 0, nsm, s, kv_stats ? &E : nullptr)) != SA_OK)
    return rc;
  if (kv_stats != nullptr) p.bypass = bypass;
  int* ticket = at<int>(ws, l.ticket);
  rc = sa::launch_select_build(p, scores, seq_lens, page_table, kp, vp, k_new, v_new, kv_stats, summaries, sel_idx,
                               sel_cnt, at<void>(ws, l.tiles), at<int>(ws, l.ntiles), status, ticket, s);
  if (rc == SA_ERR_UNSUPPORTED) {   // candidates beyond the fused kernel's capacity: two kernels
    if ((rc = sa::launch_topk(p, scores, seq_lens, sel_idx, sel_cnt, s)) != SA_OK) return rc;
    rc = sa::launch_build_step(p, seq_lens, page_table, kp, vp, k_new, v_new, kv_stats, summaries, sel_idx, sel_cnt,
                               at<void>(ws, l.tiles), at<int>(ws, l.ntiles), status, ticket, s);
  }
  if (rc != SA_OK) return rc;
  return sa::launch_decode(p, q, page_table, at<void>(ws, l.tiles), at<int>(ws, l.ntiles), at<float>(ws, l.partials),
                           ticket, out, lse, nullptr, status, tmK, tmV, nsm, s);
}

}  // namespace sa_host

extern "C" {

int sa_decode_step(const sa_problem* prob, const void* q, const void* k_pool, const void* v_pool,
                   const int32_t* page_table, const int32_t* seq_lens, void* summaries, int32_t* sel_idx,
                   int32_t* sel_cnt, float* out, float* lse, void* ws, void* stream) {
  return decode_step_impl(prob, q, nullptr, nullptr, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx,
                          sel_cnt, out, lse, ws, stream);
}

struct sa_step_plan {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

int sa_step_plan_create(const sa_problem* prob, const void* q, const void* k_pool, const void* v_pool,
                        const int32_t* page_table, const int32_t* seq_lens, void* summaries, int32_t* sel_idx,
                        int32_t* sel_cnt, float* out, float* lse, void* ws, sa_step_plan** plan) {
  if (plan == nullptr) return SA_ERR_INVALID_ARG;
  *plan = nullptr;
  // the host-visible checks first, so that a bad argument returns before any capture
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !summaries || !sel_idx || !sel_cnt || !out || !lse ||
      !ws)
    return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(summaries) || !aligned16(out) ||
      !aligned16(ws))
    return SA_ERR_INVALID_ARG;
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return SA_ERR_CUDA;
  // relaxed: a first call in the process sets kernel attributes and queries
  // occupancy while capturing
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return SA_ERR_CUDA;
  }
  rc = decode_step_impl(prob, q, nullptr, nullptr, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt,
                        out, lse, ws, cs);
  cudaGraph_t g = nullptr;
  const cudaError_t ec = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (rc != SA_OK || ec != cudaSuccess) {
    if (g != nullptr) cudaGraphDestroy(g);
    return rc != SA_OK ? rc : SA_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return SA_ERR_CUDA;
  }
  *plan = new sa_step_plan{g, ex};
  return SA_OK;
}

int sa_step_plan_launch(sa_step_plan* plan, void* stream) {
  if (plan == nullptr) return SA_ERR_INVALID_ARG;
  return cudaGraphLaunch(plan->exec, as_stream(stream)) == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int sa_step_plan_destroy(sa_step_plan* plan) {
  if (plan == nullptr) return SA_OK;
  cudaGraphExecDestroy(plan->exec);
  cudaGraphDestroy(plan->graph);
  delete plan;
  return SA_OK;
}

int sa_decode_step_append(const sa_problem* prob, const void* q, const void* k_new, const void* v_new, void* k_pool,
                          void* v_pool, const int32_t* page_table, const int32_t* seq_lens, void* summaries,
                          int32_t* sel_idx, int32_t* sel_cnt, float* out, float* lse, void* ws, void* stream) {
  if (k_new == nullptr || v_new == nullptr) return SA_ERR_INVALID_ARG;
  return decode_step_impl(prob, q, k_new, v_new, k_pool, v_pool, page_table, seq_lens, summaries, sel_idx, sel_cnt,
                          out, lse, ws, stream);
}

int sa_decode_step_bypass(const sa_problem* prob, const void* q, const void* k_new_or_null,
                          const void* v_new_or_null, void* k_pool, void* v_pool, const int32_t* page_table,
                          const int32_t* seq_lens, void* summaries, float* kv_stats, float eps, int32_t* sel_idx,
                          int32_t* sel_cnt, float* out, float* lse, float* rho_or_null, int32_t* bypass, void* ws,
                          void* stream) {
  if (kv_stats == nullptr || bypass == nullptr || !aligned16(kv_stats)) return SA_ERR_INVALID_ARG;
  return decode_step_impl(prob, q, k_new_or_null, v_new_or_null, k_pool, v_pool, page_table, seq_lens, summaries,
                          sel_idx, sel_cnt, out, lse, ws, stream, kv_stats, eps, rho_or_null, bypass);
}

int sa_kv_stats(const sa_problem* prob, const void* k_pool, const void* v_pool, const int32_t* page_table,
                const int32_t* seq_lens, float* kv_stats, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!k_pool || !v_pool || !page_table || !seq_lens || !kv_stats || !ws) return SA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(kv_stats)) return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  return sa::launch_kv_stats(p, k_pool, v_pool, page_table, seq_lens, kv_stats, at<int>(ws, l.header),
                             as_stream(stream));
}

int sa_head_sparsity(const sa_problem* prob, const void* q, const void* k_pool, const int32_t* page_table,
                     const int32_t* seq_lens, const float* kv_stats, float eps, float* rho_or_null, int32_t* bypass,
                     float* out, float* lse, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !k_pool || !page_table || !seq_lens || !kv_stats || !bypass || !out || !lse || !ws)
    return SA_ERR_INVALID_ARG;
  if (!(eps >= 0.f && eps <= 1.f)) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(kv_stats) || !aligned16(out)) return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  // without k_new the estimate reads the sums and writes nothing back
  const sa::EstArgs E{static_cast<const __nv_bfloat16*>(k_pool), page_table, nullptr, nullptr,
                      const_cast<float*>(kv_stats), eps, rho_or_null, bypass, out, lse, at<int>(ws, l.header)};
  return sa::launch_sparsity(p, q, seq_lens, E, as_stream(stream));
}

int sa_append_kv(const sa_problem* prob, const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                 const int32_t* page_table, const int32_t* seq_lens, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!k_new || !v_new || !k_pool || !v_pool || !page_table || !seq_lens || !ws) return SA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool)) return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  return sa::launch_append_kv(p, seq_lens, page_table, k_new, v_new, k_pool, v_pool, at<int>(ws, l.header),
                              as_stream(stream));
}

int sa_select_tokens(const sa_problem* prob, const void* q, const void* k_pool, const int32_t* page_table,
                     const int32_t* seq_lens, const int32_t* cand_idx, const int32_t* cand_cnt, int32_t* sel_idx,
                     int32_t* sel_cnt, float* scores_or_null, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !k_pool || !page_table || !seq_lens || !cand_idx || !cand_cnt || !sel_idx || !sel_cnt || !ws)
    return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool)) return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  return sa::launch_token_topk(p, q, k_pool, page_table, seq_lens, cand_idx, cand_cnt, sel_idx, sel_cnt,
                               scores_or_null, at<int>(ws, l.header), as_stream(stream));
}

int sa_update_score_tables(const sa_problem* prob, const float* vert_in, const float* slash_in, float* vert_out,
                           float* slash_out, const int32_t* prev_seq_lens, const int32_t* prev_sel_idx,
                           const int32_t* prev_sel_cnt, const float* prev_logits, const float* prev_lse,
                           const int32_t* prev_bypass_or_null, const int32_t* seq_lens, float decay, float beta,
                           int32_t* cand_idx, int32_t* cand_cnt, void* ws, void* stream) {
  Params p;
  int rc = make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!vert_in || !slash_in || !vert_out || !slash_out || !seq_lens || !cand_idx || !cand_cnt || !ws)
    return SA_ERR_INVALID_ARG;
  if (!(decay > 0.f && decay < 1.f) || !(beta > 0.f) || !std::isfinite(beta)) return SA_ERR_INVALID_ARG;
  const bool has_prev = prev_logits != nullptr;
  if (has_prev && (!prev_seq_lens || !prev_sel_idx || !prev_sel_cnt || !prev_lse)) return SA_ERR_INVALID_ARG;
  const size_t bytes = (size_t)p.B * p.Hq * p.mpp * SA_PAGE_SIZE * sizeof(float);
  auto overlap = [bytes](const void* a, const void* b) {
    const char* x = static_cast<const char*>(a);
    const char* y = static_cast<const char*>(b);
    return x < y + bytes && y < x + bytes;
  };
  if (overlap(vert_out, vert_in) || overlap(vert_out, slash_in) || overlap(slash_out, vert_in) ||
      overlap(slash_out, slash_in) || overlap(vert_out, slash_out))
    return SA_ERR_INVALID_ARG;
  const Layout l = layout_of(p);
  sa::TableArgs A;
  A.vin = vert_in;
  A.sin = slash_in;
  A.vout = vert_out;
  A.sout = slash_out;
  A.prev_lens = prev_seq_lens;
  A.prev_sel = prev_sel_idx;
  A.prev_cnt = prev_sel_cnt;
  A.prev_logits = prev_logits;
  A.prev_lse = prev_lse;
  A.frozen = prev_bypass_or_null;
  A.lens = seq_lens;
  A.cand = cand_idx;
  A.cand_cnt = cand_cnt;
  sa::tables_stage_ptrs(p, at<void>(ws, l.stage), &A.stage, &A.stage_cnt);
  A.status = at<int>(ws, l.header);
  A.decay = decay;
  A.beta = beta;
  return sa::launch_tables(p, A, as_stream(stream));
}

int sa_lse_merge(int32_t n_rows, int32_t D, const float* o_a, const float* lse_a, const float* o_b,
                 const float* lse_b, float* o, float* lse, void* stream) {
  if (n_rows < 0 || D < 1) return SA_ERR_INVALID_ARG;
  if (n_rows == 0) return SA_OK;
  if (!o_a || !lse_a || !o_b || !lse_b || !o || !lse) return SA_ERR_INVALID_ARG;
  return sa::launch_lse_merge(n_rows, D, o_a, lse_a, o_b, lse_b, o, lse, as_stream(stream));
}

}  // extern "C"
