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

namespace sa {

constexpr int kSumWarps = 8;

__global__ void __launch_bounds__(kSumWarps * 32)
summarize_kernel(Params p, const __nv_bfloat16* __restrict__ k_pool, const int* __restrict__ page_table,
                 const int* __restrict__ seq_lens, int block_begin, int block_end,
                 __nv_bfloat16* __restrict__ summ, int* status) {
  pdl_wait();
  pdl_trigger();
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = min(seq_lens[b], p.mpp * kP);
  const int Bs = p.bs[kvh];
  const int nblk = (L + Bs - 1) / Bs;
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
  const size_t unit_slot = ((size_t)b * p.Hk + kvh) * p.slots;

  for (int j = jb + blockIdx.x * kSumWarps + warp; j < je; j += gridDim.x * kSumWarps) {
    const int t0 = j * Bs;
    const int t1 = min(t0 + Bs, L);
    float mn[4], mx[4], sm[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) { mn[i] = INFINITY; mx[i] = -INFINITY; sm[i] = 0.f; }
    bool bad = false;
    // walk the block page by page, rows in ascending token order
    for (int t = t0; t < t1;) {
      const int lp = t / kP;
      const int row0 = t % kP;
      const int rows = min(kP - row0, t1 - t);
      const int phys = pt[lp];
      if (phys < 0 || phys >= p.num_pages) {
        bad = true;
        t += rows;
        continue;
      }
      const uint2* src = reinterpret_cast<const uint2*>(
          k_pool + (((size_t)phys * p.Hk + kvh) * kP + row0) * kD) + lane;
      uint2 v[kP];
#pragma unroll
      for (int r = 0; r < kP; ++r)
        if (r < rows) v[r] = __ldg(src + r * (kD / 4));
#pragma unroll
      for (int r = 0; r < kP; ++r) {
        if (r < rows) {
          const float x0 = bf16_lo(v[r].x), x1 = bf16_hi(v[r].x);
          const float x2 = bf16_lo(v[r].y), x3 = bf16_hi(v[r].y);
          if (p.mode == SA_SUMMARY_MINMAX) {
            mn[0] = fminf(mn[0], x0); mx[0] = fmaxf(mx[0], x0);
            mn[1] = fminf(mn[1], x1); mx[1] = fmaxf(mx[1], x1);
            mn[2] = fminf(mn[2], x2); mx[2] = fmaxf(mx[2], x2);
            mn[3] = fminf(mn[3], x3); mx[3] = fmaxf(mx[3], x3);
          } else {
            sm[0] = __fadd_rn(sm[0], x0);
            sm[1] = __fadd_rn(sm[1], x1);
            sm[2] = __fadd_rn(sm[2], x2);
            sm[3] = __fadd_rn(sm[3], x3);
          }
        }
      }
      t += rows;
    }
    if (bad) {
      if (lane == 0) set_status(status, SA_ERR_BAD_PAGE);
#pragma unroll
      for (int i = 0; i < 4; ++i) { mn[i] = mx[i] = sm[i] = 0.f; }
    }
    const int n = t1 - t0;
    if (p.mode == SA_SUMMARY_MINMAX) {
      uint2* dst = reinterpret_cast<uint2*>(summ + (unit_slot + j) * 2 * kD) + lane;
      uint2 lo, hi;
      lo.x = pack_bf16(mn[0], mn[1]); lo.y = pack_bf16(mn[2], mn[3]);
      hi.x = pack_bf16(mx[0], mx[1]); hi.y = pack_bf16(mx[2], mx[3]);
      dst[0] = lo;            // row 0: min
      dst[kD / 4] = hi;       // row 1: max
    } else {
      const float fn = (float)n;
      uint2 o;
      if (bad || n <= 0) {
        o.x = o.y = 0u;
      } else {
        o.x = pack_bf16(__fdiv_rn(sm[0], fn), __fdiv_rn(sm[1], fn));
        o.y = pack_bf16(__fdiv_rn(sm[2], fn), __fdiv_rn(sm[3], fn));
      }
      reinterpret_cast<uint2*>(summ + (unit_slot + j) * kD)[lane] = o;
    }
  }
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
