// One whole decode step in four launches: block scores (a2), per-head top-k
// (a3), then one CTA per (sequence, KV head) that builds the group's tile
// list and refreshes the summary of the block holding the newest token (a1,
// incremental), then the paged decode with the exact log-sum-exp merge
// (a4-a6).
//
// The tail block is never a candidate (it sits in the recent window, W >= Bs),
// so refreshing its summary after scoring gives the same result as before.
#include <cuda.h>

#include <algorithm>

#include "sa_common.cuh"
#include "sparsity.cuh"
#include "summary.cuh"
#include "tiles.cuh"
#include "topk.cuh"

namespace sa {

// Tile list of one window of one (sequence, KV head) by warps 0..30, and (in
// the window-0 CTA) the incremental summary of its block holding token L - 1
// by warp 31, which takes no part in the builder's barriers.
constexpr int kStepBuildThreads = 1024;
constexpr int kStepTileThreads = kStepBuildThreads - 32;

__global__ void __launch_bounds__(kStepBuildThreads)
build_step_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ page_table,
                  __nv_bfloat16* k_pool, __nv_bfloat16* v_pool, const __nv_bfloat16* __restrict__ k_new,
                  const __nv_bfloat16* __restrict__ v_new, float* stats, __nv_bfloat16* __restrict__ summ,
                  const int* sel_idx, int* sel_cnt, Tile* __restrict__ tiles, int* __restrict__ ntiles, int* status,
                  int* ticket) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) *ticket = 0;   // the decode's chunk tickets
  extern __shared__ int smem_b[];   // build_smem_bytes(mpp): window flags, then window masks
  __shared__ int scan_tmp[32];
  const int kvh = blockIdx.x, b = blockIdx.y;
  if (threadIdx.x >= kStepTileThreads) {
    if (blockIdx.z != 0) return;
    const int L = min(seq_lens[b], p.mpp * kP);
    if (k_new != nullptr) {
      append_token_warp(p, b, kvh, L, k_new, v_new, k_pool, v_pool, page_table + (size_t)b * p.mpp, status);
      if (stats != nullptr) stats_add_new_warp(p, stats, k_new, v_new, b, kvh, L);   // read by the scores only
    }
    if (L > 0)
      summarize_block_warp(p, b, kvh, (L - 1) / p.bs[kvh], L, k_pool, page_table + (size_t)b * p.mpp, summ, status);
    return;
  }
  const int win = min(p.mpp, kWinPages);
  const size_t h0 = (size_t)b * p.Hq + kvh * p.G;
  const uint32_t active = unit_active_heads(p, b, kvh);
  build_unit_tiles<kStepTileThreads>(p, b, kvh, seq_lens, page_table, sel_idx + h0 * p.kcap, sel_cnt + h0,
                                     SA_SEL_BLOCK, tiles, ntiles, status, smem_b,
                                     reinterpret_cast<uint32_t*>(smem_b + win), scan_tmp, active, blockIdx.z, 1);
  // heads answered by the sparsity bypass report no selection (the builders
  // of every window leave those heads out whatever their counts read)
  if (blockIdx.z == 0 && p.bypass != nullptr && threadIdx.x < p.G && p.bypass[h0 + threadIdx.x])
    sel_cnt[h0 + threadIdx.x] = 0;
}

int launch_build_step(const Params& p, const int* seq_lens, const int* page_table, void* k_pool, void* v_pool,
                      const void* k_new, const void* v_new, float* stats, void* summ, const int* sel_idx, int* sel_cnt,
                      void* tiles, int* ntiles, int* status, int* ticket, cudaStream_t stream) {
  const size_t smem = build_smem_bytes(p.mpp);
  // static + dynamic shared memory can pass the 48 KB default even when the
  // dynamic part alone does not: always opt in (cached per kernel)
  smem_limit_at_least(reinterpret_cast<const void*>(build_step_kernel), (int)smem);
  const cudaError_t e = launch_pdl(build_step_kernel, dim3(p.Hk, p.B, num_windows(p.mpp)), dim3(kStepBuildThreads),
                                   smem, stream, p,
                                   seq_lens, page_table, static_cast<__nv_bfloat16*>(k_pool),
                                   static_cast<__nv_bfloat16*>(v_pool), static_cast<const __nv_bfloat16*>(k_new),
                                   static_cast<const __nv_bfloat16*>(v_new), stats, static_cast<__nv_bfloat16*>(summ),
                                   sel_idx, sel_cnt, static_cast<Tile*>(tiles), ntiles, status, ticket);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

// ------------------------------------------------------------------ append

// One warp per (KV head, sequence): the new token's K and V rows at L - 1.
__global__ void __launch_bounds__(32)
append_kv_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ page_table,
                 const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new,
                 __nv_bfloat16* k_pool, __nv_bfloat16* v_pool, int* status) {
  pdl_wait();
  pdl_trigger();
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int L = min(seq_lens[b], p.mpp * kP);
  append_token_warp(p, b, kvh, L, k_new, v_new, k_pool, v_pool, page_table + (size_t)b * p.mpp, status);
}

int launch_append_kv(const Params& p, const int* seq_lens, const int* page_table, const void* k_new, const void* v_new,
                     void* k_pool, void* v_pool, int* status, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(append_kv_kernel, dim3(p.Hk, p.B), dim3(32), 0, stream, p, seq_lens, page_table,
                                   static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new),
                                   static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool), status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

// ------------------------------------------------------------------ fused

// One CTA per (sequence, KV head): the top-k of the group's G query heads
// (head g on threads [g GROUP, (g + 1) GROUP), named barrier 1 + g, the
// selections kept in shared memory), then the tile list of their union
// (warps 0..30) and the tail summary (warp 31), as build_step_kernel.  It
// replaces topk_kernel + build_step_kernel when every head's candidates fit
// GROUP x KPT keys.  GRP (group-shared selection) and APPEND (the new
// token's rows written too) are separate instantiations, so that the plain
// step's kernel carries none of their code or registers.
template <int GROUP, int KPT, bool GRP, bool APPEND>
__global__ void __launch_bounds__(kStepBuildThreads)
select_build_kernel(Params p, const float* __restrict__ scores, const int* __restrict__ seq_lens,
                    const int* __restrict__ page_table, __nv_bfloat16* k_pool, __nv_bfloat16* v_pool,
                    const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new, float* stats,
                    __nv_bfloat16* __restrict__ summ, int* __restrict__ sel_idx, int* __restrict__ sel_cnt,
                    Tile* __restrict__ tiles, int* __restrict__ ntiles, int* status, int* ticket) {
  // the call's sequence lengths are ready when this kernel starts (it is the
  // second of the step): the candidate range is read before the wait
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int L = min(seq_lens[b], p.mpp * kP);
  int j0, j1;
  candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ticket = 0;   // the decode's chunk tickets
  extern __shared__ int smem_b[];   // window flags, window masks, then selections [G][kcap] and counts [G]
  __shared__ TopkScratch S[kStepBuildThreads / GROUP];
  __shared__ int scan_tmp[32];
  const int G = p.G;
  const int win = min(p.mpp, kWinPages);
  int* s_sel = smem_b + build_smem_bytes(p.mpp) / sizeof(int);
  int* s_cnt = s_sel + G * p.kcap;
  const uint32_t active = unit_active_heads(p, b, kvh);   // loaded now, used after the top-k
  const int g = tid / GROUP;
  if (GRP) {   // one list for the group, from the summed scores
    if (g == 0)
      group_topk<GROUP, KPT, true>(scores + ((size_t)b * p.Hq + kvh * G) * p.slots + j0, j1 - j0, p.k[kvh * G], j0,
                                   s_sel, s_cnt, 1, S[0], G, (size_t)p.slots);
    __syncthreads();
    for (int i = tid; i < (G - 1) * p.kcap; i += kStepBuildThreads) s_sel[p.kcap + i] = s_sel[i % p.kcap];
    if (tid > 0 && tid < G) s_cnt[tid] = s_cnt[0];
  } else if (g < G) {
    const int h = kvh * G + g;
    group_topk<GROUP, KPT>(scores + ((size_t)b * p.Hq + h) * p.slots + j0, j1 - j0, p.k[h], j0,
                           s_sel + g * p.kcap, s_cnt + g, 1 + g, S[g]);
  }
  __syncthreads();
  const size_t h0 = (size_t)b * p.Hq + kvh * G;
  if (p.bypass != nullptr) {   // heads answered by the sparsity bypass select nothing
    if (tid < G && !((active >> tid) & 1u)) s_cnt[tid] = 0;
    __syncthreads();
  }
  if (tid >= kStepTileThreads) {
    // the selections out (the tile build reads them from shared memory and
    // starts at once), then the append and the tail summary
    const int lane = tid & 31;
    for (int gg = 0; gg < G; ++gg)
      for (int i = lane; i < s_cnt[gg]; i += 32) sel_idx[(h0 + gg) * p.kcap + i] = s_sel[gg * p.kcap + i];
    if (lane < G) sel_cnt[h0 + lane] = s_cnt[lane];
    if (APPEND) {
      append_token_warp(p, b, kvh, L, k_new, v_new, k_pool, v_pool, page_table + (size_t)b * p.mpp, status);
      if (stats != nullptr) stats_add_new_warp(p, stats, k_new, v_new, b, kvh, L);   // read by the scores only
    }
    if (L > 0)
      summarize_block_warp(p, b, kvh, (L - 1) / p.bs[kvh], L, k_pool, page_table + (size_t)b * p.mpp, summ, status);
    return;
  }
  build_unit_tiles<kStepTileThreads>(p, b, kvh, seq_lens, page_table, s_sel, s_cnt, SA_SEL_BLOCK, tiles, ntiles,
                                     status, smem_b, reinterpret_cast<uint32_t*>(smem_b + win), scan_tmp, active, 0,
                                     num_windows(p.mpp));
}

// SA_ERR_UNSUPPORTED when some head's candidates exceed the fused kernel's
// key capacity or its shared memory would not fit; the caller then runs
// topk_kernel + build_step_kernel.
int launch_select_build(const Params& p, const float* scores, const int* seq_lens, const int* page_table,
                        void* k_pool, void* v_pool, const void* k_new, const void* v_new, float* stats, void* summ,
                        int* sel_idx, int* sel_cnt, void* tiles, int* ntiles, int* status, int* ticket,
                        cudaStream_t stream) {
  const int max_n = max_candidates(p);
  const size_t smem = build_smem_bytes(p.mpp) + ((size_t)p.G * p.kcap + p.G) * sizeof(int);
  if (smem > 160 * 1024) return SA_ERR_UNSUPPORTED;
  void (*kern)(Params, const float*, const int*, const int*, __nv_bfloat16*, __nv_bfloat16*, const __nv_bfloat16*,
               const __nv_bfloat16*, float*, __nv_bfloat16*, int*, int*, Tile*, int*, int*, int*) = nullptr;
  const int v = (p.sel_mode == SA_SELECT_GROUP ? 2 : 0) | (k_new != nullptr ? 1 : 0);
#define SA_SB_PICK(GG, KK)                                                             \
  (v == 0 ? select_build_kernel<GG, KK, false, false> : v == 1 ? select_build_kernel<GG, KK, false, true> \
   : v == 2 ? select_build_kernel<GG, KK, true, false> : select_build_kernel<GG, KK, true, true>)
  if (p.G <= 4) {
    if (max_n <= 256 * 8) kern = SA_SB_PICK(256, 8);
    else if (max_n <= 256 * 16) kern = SA_SB_PICK(256, 16);
  } else {
    if (max_n <= 128 * 16) kern = SA_SB_PICK(128, 16);
  }
#undef SA_SB_PICK
  if (kern == nullptr) return SA_ERR_UNSUPPORTED;
  smem_limit_at_least(reinterpret_cast<const void*>(kern), (int)smem);
  const cudaError_t e = launch_pdl(kern, dim3(p.Hk, p.B), dim3(kStepBuildThreads), smem, stream, p, scores, seq_lens,
                                   page_table, static_cast<__nv_bfloat16*>(k_pool),
                                   static_cast<__nv_bfloat16*>(v_pool), static_cast<const __nv_bfloat16*>(k_new),
                                   static_cast<const __nv_bfloat16*>(v_new), stats, static_cast<__nv_bfloat16*>(summ),
                                   sel_idx, sel_cnt, static_cast<Tile*>(tiles), ntiles, status, ticket);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
