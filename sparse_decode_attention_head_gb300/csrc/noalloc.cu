// sa_sparse_decode_noalloc: the sparse decode step for callers that cannot
// allocate device memory.
//
// sa_sparse_decode needs a caller-allocated workspace for its scratch (the
// per-KV-head tile lists and their counts, the split-K chunk partials and
// the chunk ticket).
// Some callers cannot provide one: code that runs inside a host framework
// which owns every device allocation through its own pool and forbids any
// other cudaMalloc, or a latency-critical path where cudaMalloc's implicit
// device synchronisation is not allowed.  This entry point takes the same
// inputs and outputs but keeps its scratch in one fixed-size array in device
// global memory that belongs to this library (kNoAllocScratchBytes per GPU,
// held by every GPU that loads the library until the process exits).
//
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress (with
// that device current) and caches it with the id of the context it belongs
// to (a reset device, or another context on it, is looked up again).  Every call shares the array and it
// keeps the last call's contents: the status word is cleared at the start of
// each call (the tile builder zeroes the chunk ticket), and two calls that overlap on the
// GPU (different streams, or different host threads) race on it.
#include <cuda.h>

#include <mutex>

#include "launch.cuh"


namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;   // 64 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
// The array's device address belongs to a CUDA context, not to a device
// ordinal: after cudaDeviceReset, or under another driver-API context, the
// same ordinal has a different context and the array a different address.
// The address is therefore cached with the unique id of the context it was
// looked up in (cuCtxGetId; ids are never reused within a process).
struct ScratchEntry {
  unsigned long long ctx_id;
  void* ptr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the current context, or 0 if it cannot be had (then the
// address is looked up again on every call).
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

struct NoAllocLayout {
  size_t status, ticket, ntiles, tiles, partials, total;
};

NoAllocLayout layout_of(const sa::Params& p) {
  NoAllocLayout l;
  size_t off = 0;
  l.status = off;
  off = up256(off + sizeof(int));
  l.ticket = off;   // the decode's chunk ticket (zeroed by the tile builder)
  off = up256(off + sizeof(int));
  l.ntiles = off;   // tile counts per (unit, window)
  off = up256(off + sa::ntiles_bytes(p));
  l.tiles = off;
  off = up256(off + sa::tiles_bytes(p));
  l.partials = off;
  off = up256(off + sa::decode_partials_bytes(p));
  l.total = off;
  return l;
}

// Device address of the scratch array in the current context (looked up on
// the first call in that context, with its device current).
int scratch_on_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
  unsigned long long id = current_context_id();   // 0 before the runtime has made a context current
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchEntry& e = g_scratch[dev];
  if (e.ptr == nullptr || id == 0 || e.ctx_id != id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return SA_ERR_CUDA;
    if (id == 0) id = current_context_id();   // the lookup itself has made the context current
    e.ptr = ptr;
    e.ctx_id = id;
  }
  *out = e.ptr;
  return SA_OK;
}

inline bool aligned16(const void* x) { return (reinterpret_cast<uintptr_t>(x) & 15u) == 0; }

}  // namespace

extern "C" int sa_sparse_decode_noalloc(const sa_problem* prob, const void* q, const void* k_pool,
                                        const void* v_pool, const int32_t* page_table, const int32_t* seq_lens,
                                        const int32_t* sel_idx, const int32_t* sel_cnt, int32_t sel_granularity,
                                        float* out, float* lse, float* logits_or_null, int32_t* status_or_null,
                                        void* stream) {
  sa::Params p;
  int rc = sa_host::make_params(prob, &p);
  if (rc != SA_OK) return rc;
  if (!q || !k_pool || !v_pool || !page_table || !seq_lens || !sel_idx || !sel_cnt || !out || !lse)
    return SA_ERR_INVALID_ARG;
  if (sel_granularity != SA_SEL_BLOCK && sel_granularity != SA_SEL_TOKEN) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out)) return SA_ERR_INVALID_ARG;
  if ((size_t)p.mpp * sizeof(int) > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (sa::decode_smem_bytes(p) > 227 * 1024) return SA_ERR_UNSUPPORTED;
  const NoAllocLayout l = layout_of(p);
  if (l.total > kNoAllocScratchBytes) return SA_ERR_CAPACITY;   // problem too large for the fixed scratch
  void* base = nullptr;
  if ((rc = scratch_on_current_device(&base)) != SA_OK) return rc;
  const int nsm = sa_host::num_sms_current();
  if (nsm <= 0) return SA_ERR_CUDA;
  CUtensorMap tmK, tmV;
  if ((rc = sa_host::make_kv_map(&tmK, k_pool, p)) != SA_OK) return rc;
  if ((rc = sa_host::make_kv_map(&tmV, v_pool, p)) != SA_OK) return rc;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* b = static_cast<char*>(base);
  int* status = status_or_null ? status_or_null : reinterpret_cast<int*>(b + l.status);
  int* ticket = reinterpret_cast<int*>(b + l.ticket);
  // what must start at zero: the status word (the tile builder zeroes the
  // chunk ticket)
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return SA_ERR_CUDA;
  rc = sa::launch_build_tiles(p, seq_lens, page_table, sel_idx, sel_cnt, sel_granularity, b + l.tiles,
                              reinterpret_cast<int*>(b + l.ntiles), status, ticket, s);
  if (rc != SA_OK) return rc;
  return sa::launch_decode(p, q, page_table, b + l.tiles, reinterpret_cast<int*>(b + l.ntiles),
                           reinterpret_cast<float*>(b + l.partials), ticket, out, lse, logits_or_null, status,
                           tmK, tmV, nsm, s);
}
