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

// Bit r (r < 16) set when token t0 + r lies in [lo, hi).
__device__ __forceinline__ uint32_t token_bits(int t0, int lo, int hi) {
  const int a = min(max(lo - t0, 0), kP), b = min(max(hi - t0, 0), kP);
  return b > a ? ((1u << b) - 1u) & ~((1u << a) - 1u) : 0u;
}

// Bit j of a 4-bit value moved to bit 8 j (the four products of the
// multiplier land on distinct bits, so nothing carries).
__device__ __forceinline__ uint32_t spread_nibble(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

// G-bit mask of the unit's heads that attend: those not answered by the
// sparsity bypass (all heads when p.bypass is NULL).
__device__ __forceinline__ uint32_t unit_active_heads(const Params& p, int b, int kvh) {
  uint32_t active = (1u << p.G) - 1u;
  if (p.bypass != nullptr)
    for (int g = 0; g < p.G; ++g)
      if (p.bypass[(size_t)b * p.Hq + kvh * p.G + g]) active &= ~(1u << g);
  return active;
}

// Pages per builder window: the builder keeps a flag and 16 token masks per
// page of the current window in shared memory (20 bytes a page, plus 16 so
// that the masks can start on a 16-byte boundary).
constexpr int kWinPages = 4096;

__host__ __device__ inline size_t build_smem_bytes(int mpp) {
  const int w = mpp < kWinPages ? mpp : kWinPages;
  return (size_t)w * (sizeof(int) + 4 * sizeof(uint32_t)) + 16;
}

// A unit's tile list is kept in segments, one per window of kWinPages pages:
// the tiles of window w start at entry w * kWinPages of the unit's
// max_pages_per_seq entries, and ntiles[unit * num_windows + w] counts them.
// The windows of one unit can then be built by different CTAs.
__host__ __device__ inline int num_windows(int mpp) { return (mpp + kWinPages - 1) / kWinPages; }

// Collective over threads [0, NT) (named barrier 1): build the tile-list
// segments of windows [w_first, w_first + w_count) of unit (b, kvh).  Thread
// t owns the contiguous pages [t per, t per + per) of each window.  Every global load is issued up front (sequence length, the
// first window's page-table entries, the thread's first selection entries),
// then: dense-set masks, selected tokens OR-ed in (shared-memory atomics),
// a block scan of the page flags, and one 32-byte store per tile.
// sel_row: the unit's selections [G][kcap] (global or shared memory),
// cnt_row: their counts [G].  A page's four mask words are one 16-byte
// access (conflict-free across a warp's contiguous page ranges).  active: the heads that attend (G bits); the
// others are left out -- no tokens attend for them and their output rows are
// not written.  A unit with no tile at all (L = 0) is answered by the
// decode's merge (O = 0, lse = -inf).  s_flag: window ints, s_mask: 4 window words,
// scan_tmp: 32 ints.
template <int NT>
__device__ __forceinline__ void build_unit_tiles(const Params& p, int b, int kvh, const int* __restrict__ seq_lens,
                                                 const int* __restrict__ page_table, const int* sel_row,
                                                 const int* cnt_row, int gran, Tile* __restrict__ tiles,
                                                 int* __restrict__ ntiles, int* status, int* s_flag, uint32_t* s_mask,
                                                 int* scan_tmp, uint32_t active, int w_first, int w_count) {
  constexpr int kPer = (kWinPages + NT - 1) / NT;   // pages per thread and window, at most
  constexpr int kItemRegs = 2;                      // selection entries prefetched per thread (r = 0, 1 below)
  auto bsync = [] { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); };
  s_mask = reinterpret_cast<uint32_t*>((reinterpret_cast<uintptr_t>(s_mask) + 15) & ~uintptr_t(15));
  const int u = b * p.Hk + kvh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G;
  const int* pt_row = page_table + (size_t)b * p.mpp;
  const int win = min(p.mpp, kWinPages);
  const int per = (win + NT - 1) / NT;
  const int nwin = num_windows(p.mpp);
  const int wp_first = w_first * kWinPages;   // first page of the first window
  // ---- up-front loads (the first window's page-table entries)
  const int Lraw = seq_lens[b];
  int ptr[kPer];
#pragma unroll
  for (int r = 0; r < kPer; ++r) {
    const int i = tid * per + r;
    ptr[r] = (r < per && i < win && wp_first + i < p.mpp) ? __ldg(pt_row + wp_first + i) : -1;
  }
  const int nitems = G * p.kcap;
  int icnt[kItemRegs], iidx[kItemRegs];
#pragma unroll
  for (int r = 0; r < kItemRegs; ++r) {
    const int it = tid + r * NT;
    icnt[r] = 0;
    iidx[r] = 0;
    if (it < nitems) {
      const int g = it / p.kcap;
      icnt[r] = cnt_row[g];
      iidx[r] = sel_row[it];
    }
  }
  const int Lc = max(0, min(Lraw, p.mpp * kP));
  const int npg = (Lc + kP - 1) / kP;
  int s_end, w_beg;
  partition(Lc, p.S, p.W, s_end, w_beg);
  const int Bs = p.bs[kvh];
  const uint32_t all = active;
  Tile* T = tiles + (size_t)u * p.mpp;

  for (int wi = w_first; wi < w_first + w_count; ++wi) {
    const int w0 = wi * kWinPages;
    const int wn = max(0, min(kWinPages, npg - w0));
    if (wn == 0) {   // no page of the sequence in this window
      if (tid == 0) ntiles[u * nwin + wi] = 0;
      continue;
    }
    const int a = min(wn, tid * per), e = min(wn, a + per);
    // dense-set tokens of each page attend for every head: the page's 16-bit
    // token mask from the two dense ranges, each bit spread to a byte of `all`
    for (int i = a; i < e; ++i) {
      const int t0 = (w0 + i) * kP;
      const uint32_t tm = token_bits(t0, 0, s_end) | token_bits(t0, w_beg, Lc);
      uint32_t m[4];
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) m[w4] = spread_nibble((tm >> (4 * w4)) & 0xfu) * all;
      reinterpret_cast<uint4*>(s_mask)[i] = make_uint4(m[0], m[1], m[2], m[3]);
      s_flag[i] = tm != 0u;
    }
    bsync();
    // each head's selected tokens inside M (and inside this window)
    const int tlo = w0 * kP, thi = (w0 + wn) * kP;
    for (int it = tid, r = 0; it < nitems; it += NT, ++r) {
      const int g = it / p.kcap, i = it - g * p.kcap;
      int cnt, x;
      if (r == 0) {
        cnt = icnt[0];
        x = iidx[0];
      } else if (r == 1) {
        cnt = icnt[1];
        x = iidx[1];
      } else {
        cnt = cnt_row[g];
        x = sel_row[it];
      }
      if (i >= min(cnt, p.kcap) || !((active >> g) & 1u)) continue;
      int lo, hi;
      item_range(gran, x, Bs, Lc, s_end, w_beg, lo, hi);
      lo = max(lo, tlo);
      hi = min(hi, thi);
      for (int tok = lo; tok < hi;) {
        const int pg = tok / kP - w0;
        const int r0 = tok % kP;
        const int r1 = min(kP, r0 + (hi - tok));
        for (int w4 = r0 >> 2; w4 <= (r1 - 1) >> 2; ++w4) {
          uint32_t m = 0;
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int row = 4 * w4 + rr;
            if (row >= r0 && row < r1) m |= (1u << g) << (8 * rr);
          }
          atomicOr(&s_mask[4 * pg + w4], m);
        }
        s_flag[pg] = 1;
        tok += r1 - r0;
      }
    }
    bsync();
    // exclusive scan of the page flags over the threads' contiguous ranges
    int c = 0;
    for (int i = a; i < e; ++i) c += s_flag[i];
    const int x = warp_incl_scan(c);
    if (lane == 31) scan_tmp[warp] = x;
    bsync();
    if (warp == 0) {
      const int y = warp_incl_scan(lane < NT / 32 ? scan_tmp[lane] : 0);
      if (lane < NT / 32) scan_tmp[lane] = y;
    }
    bsync();
    int idx = w0 + (warp > 0 ? scan_tmp[warp - 1] : 0) + x - c;   // the window's segment starts at entry w0
    // one 32-byte descriptor per tile (the page-table entry prefetched when possible)
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
      const int i = a + r;
      if (r < per && i < e && s_flag[i]) {
        const int ph = wi == w_first ? ptr[r] : __ldg(pt_row + w0 + i);
        const bool ok = ph >= 0 && ph < p.num_pages;
        if (!ok) set_status(status, SA_ERR_BAD_PAGE);
        int4* dst = reinterpret_cast<int4*>(T + idx);
        dst[0] = make_int4(w0 + i, ok ? ph : -1, 0, 0);
        const uint4 mv = reinterpret_cast<const uint4*>(s_mask)[i];
        dst[1] = make_int4((int)mv.x, (int)mv.y, (int)mv.z, (int)mv.w);
        ++idx;
      }
    }
    if (tid == 0) ntiles[u * nwin + wi] = scan_tmp[NT / 32 - 1];
    bsync();   // the window's shared state is reused by the next window
  }
}

}  // namespace sa
