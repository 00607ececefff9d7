// One block summary, computed by one warp (min/max bounding box, or mean
// key in fp32 ascending-token order with IEEE division and RNE to bf16).
#pragma once

#include "sa_common.cuh"

namespace sa {

// Warp-collective: summary of block j of (b, kvh) over tokens [j Bs, min((j+1) Bs, L)).
// Plain (coherent) loads, no __restrict__: in a decode step the same kernel
// may have just written the block's newest row (append_token_warp).
__device__ __forceinline__ void summarize_block_warp(const Params& p, int b, int kvh, int j, int L,
                                                     const __nv_bfloat16* k_pool,
                                                     const int* __restrict__ pt, __nv_bfloat16* __restrict__ summ,
                                                     int* status) {
  const int lane = threadIdx.x & 31;
  const int Bs = p.bs[kvh];
  const size_t unit_slot = ((size_t)b * p.Hk + kvh) * p.slots;
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
      if (r < rows) v[r] = src[r * (kD / 4)];
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

// Warp-collective: write the new token's key and value rows (k_new / v_new
// [B][Hk][D] bf16) at position L - 1 of (b, kvh), through the page table.
// The warp's later reads of the row (the tail summary) see the writes.
__device__ __forceinline__ void append_token_warp(const Params& p, int b, int kvh, int L,
                                                  const __nv_bfloat16* __restrict__ k_new,
                                                  const __nv_bfloat16* __restrict__ v_new, __nv_bfloat16* k_pool,
                                                  __nv_bfloat16* v_pool, const int* __restrict__ pt, int* status) {
  const int lane = threadIdx.x & 31;
  if (L <= 0) return;
  const int t = L - 1;
  const int phys = pt[t / kP];
  if (phys < 0 || phys >= p.num_pages) {
    if (lane == 0) set_status(status, SA_ERR_BAD_PAGE);
    return;
  }
  const size_t src = ((size_t)b * p.Hk + kvh) * kD;
  const size_t dst = (((size_t)phys * p.Hk + kvh) * kP + t % kP) * kD;
  reinterpret_cast<uint2*>(k_pool + dst)[lane] = reinterpret_cast<const uint2*>(k_new + src)[lane];
  reinterpret_cast<uint2*>(v_pool + dst)[lane] = reinterpret_cast<const uint2*>(v_new + src)[lane];
  __syncwarp();
}

}  // namespace sa
