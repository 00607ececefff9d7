// Tile lists for the paged decode: the union over a KV head's query heads of
// the pages to read, one 16-token page per tile with a G-bit head mask per
// token (dense-set tokens for every head, selected tokens for their heads).
#pragma once

#include "sa_common.cuh"

namespace sa {

struct __align__(16) Tile {
  int lp;            // logical page
  int phys;          // physical page (page_table lookup), -1 if outside the pool
  int pad[2];
  uint32_t mask[4];  // byte i = G-bit mask of heads attending token 16 lp + i
};

// Token range [lo, hi) of a selection entry, clipped to M; empty if none.
__device__ __forceinline__ void item_range(int gran, int x, int Bs, int Lc, int s_end, int w_beg, int& lo,
                                           int& hi) {
  if (gran == SA_SEL_BLOCK) {
    if (x < 0 || Lc <= 0 || x > (Lc - 1) / Bs) { lo = hi = 0; return; }
    lo = max(x * Bs, s_end);
    hi = min((x + 1) * Bs, w_beg);
  } else {
    lo = max(x, s_end);
    hi = min(x + 1, w_beg);
  }
}

// Block-collective: build the tile list of unit (b, kvh).  `flag` is
// shared memory of max_pages_per_seq ints, `scan_tmp` 32 ints.
__device__ __forceinline__ void build_unit_tiles(const Params& p, int b, int kvh, const int* __restrict__ seq_lens,
                                                 const int* __restrict__ page_table,
                                                 const int* sel_idx, const int* sel_cnt,
                                                 int gran, Tile* __restrict__ tiles, int* __restrict__ ntiles,
                                                 float* __restrict__ out, float* __restrict__ lse, int* status,
                                                 int* flag, int* scan_tmp) {
  const int u = b * p.Hk + kvh;
  const int tid = threadIdx.x;
  const int G = p.G;
  const int Lc = max(0, min(seq_lens[b], p.mpp * kP));
  const int npg = (Lc + kP - 1) / kP;
  int s_end, w_beg;
  partition(Lc, p.S, p.W, s_end, w_beg);
  const int Bs = p.bs[kvh];
  Tile* T = tiles + (size_t)u * p.mpp;

  for (int i = tid; i < npg; i += blockDim.x) {
    const int t0 = i * kP, t1 = t0 + kP;
    flag[i] = (t0 < s_end) || (t1 > w_beg);   // page meets I
  }
  __syncthreads();
  const int nitems = G * p.kcap;
  for (int it = tid; it < nitems; it += blockDim.x) {
    const int g = it / p.kcap, i = it % p.kcap;
    const int h = kvh * G + g;
    const int cnt = min(sel_cnt[(size_t)b * p.Hq + h], p.kcap);
    if (i >= cnt) continue;
    int lo, hi;
    item_range(gran, sel_idx[((size_t)b * p.Hq + h) * p.kcap + i], Bs, Lc, s_end, w_beg, lo, hi);
    for (int pg = lo / kP; lo < hi && pg <= (hi - 1) / kP; ++pg) flag[pg] = 1;
  }
  __syncthreads();

  // exclusive scan of the page flags -> tile index (contiguous ranges per thread)
  const int per = (npg + blockDim.x - 1) / blockDim.x;
  const int a = min(npg, tid * per), e = min(npg, a + per);
  int c = 0;
  for (int i = a; i < e; ++i) c += flag[i];
  int x = c;
  const int lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scan_tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scan_tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) scan_tmp[lane] = w;
  }
  __syncthreads();
  int base = (warp > 0 ? scan_tmp[warp - 1] : 0) + x - c;
  const int total = scan_tmp[nw - 1];
  const uint32_t all = (1u << G) - 1u;
  for (int i = a; i < e; ++i) {
    if (flag[i]) flag[i] = base++;
    else flag[i] = -1;
  }
  __syncthreads();
  // descriptors: page-table loads of 4 pages are in flight together
  for (int i0 = tid; i0 < npg; i0 += 4 * blockDim.x) {
    int ph[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + k * blockDim.x;
      ph[k] = (i < npg && flag[i] >= 0) ? __ldg(page_table + (size_t)b * p.mpp + i) : 0;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = i0 + k * blockDim.x;
      if (i < npg && flag[i] >= 0) {
        Tile t;
        t.lp = i;
        const bool ok = ph[k] >= 0 && ph[k] < p.num_pages;
        if (!ok) set_status(status, SA_ERR_BAD_PAGE);
        t.phys = ok ? ph[k] : -1;
        t.pad[0] = t.pad[1] = 0;
        // dense-set tokens of this page attend for every head
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) {
          uint32_t m = 0;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int tok = i * kP + 4 * w4 + r;
            if (tok < Lc && (tok < s_end || tok >= w_beg)) m |= all << (8 * r);
          }
          t.mask[w4] = m;
        }
        T[flag[i]] = t;
      }
    }
  }
  __syncthreads();

  // OR in each head's selected tokens inside M
  for (int it = tid; it < nitems; it += blockDim.x) {
    const int g = it / p.kcap, i = it % p.kcap;
    const int h = kvh * G + g;
    const int cnt = min(sel_cnt[(size_t)b * p.Hq + h], p.kcap);
    if (i >= cnt) continue;
    int lo, hi;
    item_range(gran, sel_idx[((size_t)b * p.Hq + h) * p.kcap + i], Bs, Lc, s_end, w_beg, lo, hi);
    for (int tok = lo; tok < hi;) {
      const int pg = tok / kP;
      const int r0 = tok % kP;
      const int r1 = min(kP, r0 + (hi - tok));
      Tile* t = T + flag[pg];
      // rows [r0, r1) of this page get bit g
      for (int w4 = r0 >> 2; w4 <= (r1 - 1) >> 2; ++w4) {
        uint32_t m = 0;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int row = 4 * w4 + r;
          if (row >= r0 && row < r1) m |= (1u << g) << (8 * r);
        }
        atomicOr(&t->mask[w4], m);
      }
      tok += r1 - r0;
    }
  }
  if (tid == 0) ntiles[u] = total;
  if (total == 0) {   // nothing attended (L = 0): O = 0, lse = -inf; the decode kernel skips the unit
    for (int i = tid; i < G * kD; i += blockDim.x) out[((size_t)b * p.Hq + kvh * G) * kD + i] = 0.f;
    if (tid < G) lse[(size_t)b * p.Hq + kvh * G + tid] = -INFINITY;
  }
}

}  // namespace sa
