// The canonical fp32 block score of up to four query heads against one block
// summary, computed by the 8 lanes of a lane group (lane part p owns dims
// [16p, 16p + 16)): each lane sums its exact bf16 x bf16 products in
// ascending dim order with one rounding per step, then a butterfly over the
// parts at partner distances 4, 2, 1, then + 0.0.  The same order as the
// score kernel (select.cu), so the selections built on it are bit-identical.
#pragma once

#include "sa_common.cuh"

namespace sa {

// q of four heads for this lane's 16 dims (packed bf16 pairs) and, for
// min/max summaries, the byte selectors that pick kmax where q >= 0 and kmin
// elsewhere.
struct QSet4 {
  uint32_t qw[4][8];
  uint32_t selw[4][8];
};

// q rows [G][kD] bf16 (16-byte aligned); heads hs*4 .. hs*4 + 3, those
// beyond G repeat head 0 (their scores are discarded).
__device__ __forceinline__ void qset_load(QSet4& s, const void* q_rows, int hs, int G, int part) {
  const uint4* qs = reinterpret_cast<const uint4*>(q_rows);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int g = hs * 4 + e;
    const int gg = g < G ? g : 0;
    const uint4 a = qs[gg * (kD / 8) + 2 * part], c = qs[gg * (kD / 8) + 2 * part + 1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) {
      s.qw[e][k2] = w[k2];
      const bool p0 = bf16_lo(w[k2]) >= 0.f, p1 = bf16_hi(w[k2]) >= 0.f;
      // result bytes 0,1 from kmax (0,1) or kmin (4,5); bytes 2,3 from kmax (2,3) or kmin (6,7)
      s.selw[e][k2] = (p0 ? 0x10u : 0x54u) | (p1 ? 0x3200u : 0x7600u);
    }
  }
}

// This lane's partial sums of the four heads over one summary row (MINMAX:
// [2][kD] min then max; MEAN: [kD]).
template <int MODE>
__device__ __forceinline__ void dot4_part(const QSet4& s, const void* row, int part, float (&acc)[4]) {
  const uint4* base = reinterpret_cast<const uint4*>(row) + 2 * part;
  uint32_t xmin[8], xmax[8];
  const uint4 lo0 = base[0], lo1 = base[1];
  if (MODE == SA_SUMMARY_MINMAX) {
    const uint4 hi0 = base[kD / 8], hi1 = base[kD / 8 + 1];
    xmin[0] = lo0.x; xmin[1] = lo0.y; xmin[2] = lo0.z; xmin[3] = lo0.w;
    xmin[4] = lo1.x; xmin[5] = lo1.y; xmin[6] = lo1.z; xmin[7] = lo1.w;
    xmax[0] = hi0.x; xmax[1] = hi0.y; xmax[2] = hi0.z; xmax[3] = hi0.w;
    xmax[4] = hi1.x; xmax[5] = hi1.y; xmax[6] = hi1.z; xmax[7] = hi1.w;
  } else {
    xmax[0] = lo0.x; xmax[1] = lo0.y; xmax[2] = lo0.z; xmax[3] = lo0.w;
    xmax[4] = lo1.x; xmax[5] = lo1.y; xmax[6] = lo1.z; xmax[7] = lo1.w;
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) xmin[k2] = 0u;
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    float a = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) {
      const uint32_t w = (MODE == SA_SUMMARY_MINMAX) ? __byte_perm(xmax[k2], xmin[k2], s.selw[e][k2]) : xmax[k2];
      // fma with c = -0 is the plain product, zero signs included
      a = fma_bf16_lo(s.qw[e][k2], w, k2 == 0 ? -0.0f : a);
      a = fma_bf16_hi(s.qw[e][k2], w, a);
    }
    acc[e] = a;
  }
}

// Butterfly over the 8 parts of a lane group with the four heads spread over
// the lanes: at partner distance 4 a lane keeps two heads and sends the other
// two, at distance 2 it keeps one, at distance 1 both partners hold the same
// head.  Every add is (own partial) + (partner's partial) of one head: the
// sums of the plain per-head butterfly.  Lanes with an even part return the
// score of head (part >> 1) of the set.
__device__ __forceinline__ float butterfly4(const float (&acc)[4], int part) {
  const bool b2 = (part & 4) != 0, b1 = (part & 2) != 0;
  const float r0 = __shfl_xor_sync(0xffffffffu, b2 ? acc[0] : acc[2], 4);
  const float r1 = __shfl_xor_sync(0xffffffffu, b2 ? acc[1] : acc[3], 4);
  const float x0 = __fadd_rn(b2 ? acc[2] : acc[0], r0);   // head 2 b2
  const float x1 = __fadd_rn(b2 ? acc[3] : acc[1], r1);   // head 2 b2 + 1
  const float r2 = __shfl_xor_sync(0xffffffffu, b1 ? x0 : x1, 2);
  const float y = __fadd_rn(b1 ? x1 : x0, r2);            // head 2 b2 + b1
  const float z = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, 1));
  return __fadd_rn(z, 0.0f);
}

}  // namespace sa
