// One whole decode step in three launches: block scores (a2), then one CTA
// per (sequence, KV head) that selects the top-k blocks of the group's G
// heads (a3), builds the group's tile list and refreshes the summary of the
// block holding the newest token (a1, incremental), then the paged decode
// with the exact log-sum-exp merge (a4-a6).
//
// The tail block is never a candidate (it sits in the recent window, W >= Bs),
// so refreshing its summary after scoring gives the same result as before.
#include <cuda.h>

#include <algorithm>

#include "sa_common.cuh"
#include "summary.cuh"
#include "tiles.cuh"
#include "topk.cuh"

namespace sa {

constexpr int kSelThreads = 1024;
constexpr int kSelGroup = 256;                          // threads per head
constexpr int kSelGroups = kSelThreads / kSelGroup;     // heads selected at once
constexpr int kSelKpt = 8;                              // keys per thread
constexpr int kSelMaxCand = kSelGroup * kSelKpt;        // 2048 candidates per head

__global__ void __launch_bounds__(kSelThreads)
select_build_kernel(Params p, const float* __restrict__ scores, const int* __restrict__ seq_lens,
                    const int* __restrict__ page_table, const __nv_bfloat16* __restrict__ k_pool,
                    __nv_bfloat16* __restrict__ summ, int* sel_idx, int* sel_cnt, Tile* __restrict__ tiles,
                    int* __restrict__ ntiles, float* __restrict__ out, float* __restrict__ lse, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int flag[];   // [mpp] for the tile builder
  __shared__ int scan_tmp[32];
  __shared__ TopkScratch S[kSelGroups];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int G = p.G;
  const int L = min(seq_lens[b], p.mpp * kP);
  const int Bs = p.bs[kvh];
  int j0, j1;
  candidate_range(L, p.S, p.W, Bs, j0, j1);
  const int group = threadIdx.x / kSelGroup;
  for (int g0 = 0; g0 < G; g0 += kSelGroups) {
    const int g = g0 + group;
    if (g < G) {
      const int h = kvh * G + g;
      group_topk<kSelGroup, kSelKpt>(scores + ((size_t)b * p.Hq + h) * p.slots + j0, j1 - j0, p.k[h], j0,
                                     sel_idx + ((size_t)b * p.Hq + h) * p.kcap, sel_cnt + (size_t)b * p.Hq + h,
                                     1 + group, S[group]);
    }
    __syncthreads();
  }
  if (threadIdx.x < 32 && L > 0)   // incremental summary of the block holding token L - 1
    summarize_block_warp(p, b, kvh, (L - 1) / Bs, L, k_pool, page_table + (size_t)b * p.mpp, summ, status);
  build_unit_tiles(p, b, kvh, seq_lens, page_table, sel_idx, sel_cnt, SA_SEL_BLOCK, tiles, ntiles, out, lse, status,
                   flag, scan_tmp);
}

int select_build_max_candidates() { return kSelMaxCand; }

int launch_select_build(const Params& p, const float* scores, const int* seq_lens, const int* page_table,
                        const void* k_pool, void* summ, int* sel_idx, int* sel_cnt, void* tiles, int* ntiles,
                        float* out, float* lse, int* status, cudaStream_t stream) {
  const size_t smem = (size_t)p.mpp * sizeof(int);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(select_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const cudaError_t e = launch_pdl(select_build_kernel, dim3(p.Hk, p.B), dim3(kSelThreads), smem, stream, p, scores,
                                   seq_lens, page_table, static_cast<const __nv_bfloat16*>(k_pool),
                                   static_cast<__nv_bfloat16*>(summ), sel_idx, sel_cnt, static_cast<Tile*>(tiles),
                                   ntiles, out, lse, status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
