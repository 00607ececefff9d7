// Step a1: per-block key summaries (min/max bounding box, or mean key).
//
// The pages use block-level selection with a head-specific block size
// (Fluxion, core claim and Fig. 5) but never define the block summary; this
// kernel builds the two kinds the selection step can score: the per-dim
// min/max of the block's keys (exact in bf16) and the per-dim mean
// (fp32 sum in ascending token order, IEEE division, round-to-nearest-even).
//
// One warp per block.  Lane l owns dims [4l, 4l+4) (8 bytes of each 256-byte
// key row), so every row load of the warp is one coalesced 256-byte access;
// rows are walked in ascending token order, following the page table page by
// page.  HBM-bound: K is read once, the summary written once.
#include "sa_common.cuh"
#include "summary.cuh"

namespace sa {

constexpr int kSumWarps = 8;

__global__ void __launch_bounds__(kSumWarps * 32)
summarize_kernel(Params p, const __nv_bfloat16* __restrict__ k_pool, const int* __restrict__ page_table,
                 const int* __restrict__ seq_lens, int block_begin, int block_end,
                 __nv_bfloat16* __restrict__ summ, int* status) {
  pdl_wait();
  pdl_trigger();
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int L = min(seq_lens[b], p.mpp * kP);
  const int nblk = (L + p.bs[kvh] - 1) / p.bs[kvh];
  int jb, je;
  if (block_begin == SA_BLOCKS_TAIL) {
    jb = nblk - 1;
    je = nblk;
  } else {
    jb = block_begin;
    je = block_end < 0 ? nblk : min(block_end, nblk);
  }
  jb = max(jb, 0);
  je = min(je, p.slots);
  const int* pt = page_table + (size_t)b * p.mpp;

  for (int j = jb + blockIdx.x * kSumWarps + warp; j < je; j += gridDim.x * kSumWarps)
    summarize_block_warp(p, b, kvh, j, L, k_pool, pt, summ, status);
}

int launch_summarize(const Params& p, const void* k_pool, const int* page_table, const int* seq_lens,
                     int block_begin, int block_end, void* summ, int* status, cudaStream_t stream) {
  int span;
  if (block_begin == SA_BLOCKS_TAIL) {
    span = 1;
  } else {
    const int hi = block_end < 0 ? p.slots : min(block_end, p.slots);
    span = max(0, hi - max(block_begin, 0));
  }
  if (span == 0) return SA_OK;
  int gx = (span + kSumWarps - 1) / kSumWarps;
  gx = min(gx, 65535);   // the warp loop covers any remainder
  dim3 grid(gx, p.Hk, p.B);
  const cudaError_t e = launch_pdl(summarize_kernel, grid, dim3(kSumWarps * 32), 0, stream, p,
                                   static_cast<const __nv_bfloat16*>(k_pool), page_table, seq_lens, block_begin,
                                   block_end, static_cast<__nv_bfloat16*>(summ), status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
