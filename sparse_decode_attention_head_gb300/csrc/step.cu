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

// Tile list of one (sequence, KV head) plus the incremental summary of its
// block holding token L - 1 (warp 0 does the summary first, the rest of the
// block starts on the tile list meanwhile).
constexpr int kStepBuildThreads = 1024;

__global__ void __launch_bounds__(kStepBuildThreads)
build_step_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ page_table,
                  const __nv_bfloat16* __restrict__ k_pool, __nv_bfloat16* __restrict__ summ, const int* sel_idx,
                  const int* sel_cnt, Tile* __restrict__ tiles, int* __restrict__ ntiles, float* __restrict__ out,
                  float* __restrict__ lse, int* status, int* ticket) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *ticket = 0;   // the decode's chunk tickets
  extern __shared__ int flag[];   // [mpp] for the tile builder
  __shared__ int scan_tmp[32];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int L = min(seq_lens[b], p.mpp * kP);
  if (threadIdx.x < 32 && L > 0)
    summarize_block_warp(p, b, kvh, (L - 1) / p.bs[kvh], L, k_pool, page_table + (size_t)b * p.mpp, summ, status);
  build_unit_tiles(p, b, kvh, seq_lens, page_table, sel_idx, sel_cnt, SA_SEL_BLOCK, tiles, ntiles, out, lse, status,
                   flag, scan_tmp);
}

int launch_build_step(const Params& p, const int* seq_lens, const int* page_table, const void* k_pool, void* summ,
                      const int* sel_idx, const int* sel_cnt, void* tiles, int* ntiles, float* out, float* lse,
                      int* status, int* ticket, cudaStream_t stream) {
  const size_t smem = (size_t)p.mpp * sizeof(int);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const cudaError_t e = launch_pdl(build_step_kernel, dim3(p.Hk, p.B), dim3(kStepBuildThreads), smem, stream, p,
                                   seq_lens, page_table, static_cast<const __nv_bfloat16*>(k_pool),
                                   static_cast<__nv_bfloat16*>(summ), sel_idx, sel_cnt, static_cast<Tile*>(tiles),
                                   ntiles, out, lse, status, ticket);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
