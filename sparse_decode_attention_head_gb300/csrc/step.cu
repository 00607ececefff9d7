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
#include "summary.cuh"
#include "tiles.cuh"

namespace sa {

// Tile list of one (sequence, KV head) by warps 0..30, and the incremental
// summary of its block holding token L - 1 by warp 31, which takes no part
// in the builder's barriers.
constexpr int kStepBuildThreads = 1024;
constexpr int kStepTileThreads = kStepBuildThreads - 32;

__global__ void __launch_bounds__(kStepBuildThreads)
build_step_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ page_table,
                  const __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ summ, const int* sel_idx,
                  const int* sel_cnt, Tile* __restrict__ tiles, int* __restrict__ ntiles, float* __restrict__ out,
                  float* __restrict__ lse, int* status, int* ticket) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ticket = 0;   // the decode's chunk tickets
  extern __shared__ int smem_b[];   // build_smem_bytes(mpp): window flags, then window masks
  __shared__ int scan_tmp[32];
  const int kvh = blockIdx.x, b = blockIdx.y;
  if (threadIdx.x >= kStepTileThreads) {
    const int L = min(seq_lens[b], p.mpp * kP);
    if (L > 0)
      summarize_block_warp(p, b, kvh, (L - 1) / p.bs[kvh], L, k_pool, page_table + (size_t)b * p.mpp, summ, status);
    return;
  }
  const int win = min(p.mpp, kWinPages);
  build_unit_tiles<kStepTileThreads>(p, b, kvh, seq_lens, page_table, sel_idx, sel_cnt, SA_SEL_BLOCK, tiles, ntiles,
                                     out, lse, status, smem_b, reinterpret_cast<uint32_t*>(smem_b + win), scan_tmp);
}

int launch_build_step(const Params& p, const int* seq_lens, const int* page_table, const void* k_pool, void* summ,
                      const int* sel_idx, const int* sel_cnt, void* tiles, int* ntiles, float* out, float* lse,
                      int* status, int* ticket, cudaStream_t stream) {
  const size_t smem = build_smem_bytes(p.mpp);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const cudaError_t e = launch_pdl(build_step_kernel, dim3(p.Hk, p.B), dim3(kStepBuildThreads), smem, stream, p,
                                   seq_lens, page_table, static_cast<const __nv_bfloat16*>(k_pool),
                                   static_cast<__nv_bfloat16*>(summ), sel_idx, sel_cnt, static_cast<Tile*>(tiles),
                                   ntiles, out, lse, status, ticket);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
