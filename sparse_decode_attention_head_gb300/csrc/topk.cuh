// Top-k for one head over its candidate blocks: keep the k best by (score
// descending, block index ascending), reported ascending.  A group of GROUP
// threads (a whole block, or a slice of one with its own named barrier)
// holds KPT consecutive keys per thread in registers, finds the k-th key by
// an MSB-first radix select over order-preserving uint32 keys (starting below
// the bits every key shares; once the bucket holding the k-th key has at most
// 32 keys, one warp finds the k-th key among them directly), and compacts in
// index order.
#pragma once

#include <algorithm>

#include "sa_common.cuh"

namespace sa {

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void group_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}


// The most candidate blocks any head can have: candidates end where the
// recent window begins, at ceil(max(L - W, S) / Bs) <= ceil(max(mpp P - W, S) / Bs).
inline int max_candidates(const Params& p) {
  int m = 0;
  for (int h = 0; h < p.Hk; ++h) {
    const int w_beg = std::max(p.mpp * kP - p.W, std::min(p.S, p.mpp * kP));
    m = std::max(m, (w_beg + p.bs[h] - 1) / p.bs[h]);
  }
  return m;
}

struct TopkScratch {
  int hist[256];
  int red[2][32];
  uint32_t cand[32];   // keys of a small last bucket
  uint32_t prefix;
  int krem;
  int bcnt;            // keys in the bucket holding the k-th key
  int eqt;             // keys equal to the k-th key (from the small-bucket rank)
  int nc;              // keys gathered into cand
};

// Exclusive scan over the group; tmp holds >= GROUP / 32 ints.
template <int GROUP>
__device__ __forceinline__ int group_excl_scan(int v, int* tmp, int bar_id) {
  const int tg = threadIdx.x % GROUP, lane = tg & 31, w = tg >> 5;
  const int x = warp_incl_scan(v);
  if (lane == 31) tmp[w] = x;
  group_sync(bar_id, GROUP);
  int before = x - v;
  for (int i = 0; i < w; ++i) before += tmp[i];
  group_sync(bar_id, GROUP);
  return before;
}

// Group-collective.  sc: the head's candidate scores (n of them, block ids
// base_idx + i); with ROWS the key of block i is the fp32 sum, in row order,
// of sc[r * row_stride + i] over nrows rows (a selection shared by a KV
// head's query heads) -- a separate instantiation, so that the one-row case
// keeps its loads independent of each other.  k_req: blocks to keep.  Writes
// out[0..) and *cnt_out.
template <int GROUP, int KPT, bool ROWS = false>
__device__ void group_topk(const float* __restrict__ sc, int n, int k_req, int base_idx, int* __restrict__ out,
                           int* __restrict__ cnt_out, int bar_id, TopkScratch& S, int nrows = 1,
                           size_t row_stride = 0) {
  const int tg = threadIdx.x % GROUP, lane = tg & 31, w = tg >> 5;
  const int k = min(k_req, n);
  if (k >= n || k <= 0) {   // keep every candidate (100 % budget, or none) / keep none
    const int m = k >= n ? n : 0;
    for (int i = tg; i < m; i += GROUP) out[i] = base_idx + i;
    if (tg == 0) *cnt_out = m;
    return;
  }
  uint32_t key[KPT];
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  // a thread's KPT consecutive scores as 16-byte loads when the row allows it
  const bool vec = !ROWS && KPT % 4 == 0 && (reinterpret_cast<uintptr_t>(sc) & 15) == 0 && tg * KPT + KPT <= n;
  if (vec) {
#pragma unroll
    for (int v = 0; v < KPT / 4; ++v) {
      const float4 f = *reinterpret_cast<const float4*>(sc + tg * KPT + 4 * v);
      key[4 * v] = order_key(f.x);
      key[4 * v + 1] = order_key(f.y);
      key[4 * v + 2] = order_key(f.z);
      key[4 * v + 3] = order_key(f.w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int i = tg * KPT + q;
      float x = 0.f;
      if (i < n) {
        x = sc[i];
        if (ROWS)
          for (int r = 1; r < nrows; ++r) x = __fadd_rn(x, sc[r * row_stride + i]);
      }
      key[q] = i < n ? order_key(x) : 0u;
    }
  }
#pragma unroll
  for (int q = 0; q < KPT; ++q)
    if (tg * KPT + q < n) { kmin = min(kmin, key[q]); kmax = max(kmax, key[q]); }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    kmin = min(kmin, __shfl_xor_sync(0xffffffffu, kmin, o));
    kmax = max(kmax, __shfl_xor_sync(0xffffffffu, kmax, o));
  }
  if (lane == 0) { S.red[0][w] = (int)kmin; S.red[1][w] = (int)kmax; }
  group_sync(bar_id, GROUP);
  uint32_t gmin = 0xffffffffu, gmax = 0u;
  for (int i = 0; i < GROUP / 32; ++i) { gmin = min(gmin, (uint32_t)S.red[0][i]); gmax = max(gmax, (uint32_t)S.red[1][i]); }
  group_sync(bar_id, GROUP);
  const int common = gmin == gmax ? 32 : __clz(gmin ^ gmax);   // leading bits shared by every key
  uint32_t mask = common >= 32 ? 0xffffffffu : (common == 0 ? 0u : (0xffffffffu << (32 - common)));
  uint32_t prefix = gmin & mask;
  int krem = k;
  int eq_total = common >= 32 ? n : -1;   // keys equal to the k-th key, once known
  for (int top = 32 - common; top > 0; top -= 8) {   // this pass resolves bits [shift, top)
    const int shift = max(0, top - 8);
    const uint32_t dmask = (1u << (top - shift)) - 1u;
    for (int i = tg; i < 256; i += GROUP) S.hist[i] = 0;
    group_sync(bar_id, GROUP);
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int i = tg * KPT + q;
      if (i < n && (key[q] & mask) == prefix) atomicAdd(&S.hist[(key[q] >> shift) & dmask], 1);
    }
    group_sync(bar_id, GROUP);
    if (w == 0) {
      // lane l owns digits 255-8l .. 248-8l (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { cnt[q] = S.hist[255 - 8 * lane - q]; tot += cnt[q]; }
      const int incl = warp_incl_scan(tot);
      int above = incl - tot;
      if (above < krem && krem <= incl) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (above < krem && krem <= above + cnt[q]) {
            S.prefix = prefix | ((uint32_t)(255 - 8 * lane - q) << shift);
            S.krem = krem - above;
            S.bcnt = cnt[q];
          }
          above += cnt[q];
        }
      }
    }
    if (tg == 0) S.nc = 0;
    group_sync(bar_id, GROUP);
    prefix = S.prefix;
    krem = S.krem;
    eq_total = shift == 0 ? S.bcnt : -1;   // a pass that resolves the last bits leaves the equal keys
    mask |= dmask << shift;
    if (shift > 0 && S.bcnt <= 32) {
      // gather the bucket and let warp 0 rank its keys: the krem-th largest is T
#pragma unroll
      for (int q = 0; q < KPT; ++q) {
        const int i = tg * KPT + q;
        if (i < n && (key[q] & mask) == prefix) S.cand[atomicAdd(&S.nc, 1)] = key[q];
      }
      group_sync(bar_id, GROUP);
      if (w == 0) {
        const int nc = S.nc;
        const uint32_t mine = lane < nc ? S.cand[lane] : 0u;
        int gt_cnt = 0, ge_cnt = 0;
        for (int j = 0; j < nc; ++j) {
          const uint32_t o = __shfl_sync(0xffffffffu, mine, j);
          gt_cnt += o > mine;
          ge_cnt += o >= mine;
        }
        if (lane < nc && gt_cnt < krem && krem <= ge_cnt) {   // every lane holding T agrees
          S.prefix = mine;
          S.krem = krem - gt_cnt;
          S.eqt = ge_cnt - gt_cnt;
        }
      }
      group_sync(bar_id, GROUP);
      prefix = S.prefix;
      krem = S.krem;
      eq_total = S.eqt;
      mask = 0xffffffffu;
      group_sync(bar_id, GROUP);
      break;
    }
    group_sync(bar_id, GROUP);
  }
  const uint32_t T = prefix;   // key of the k-th best
  const int need_eq = krem;    // keys equal to T that are taken, lowest index first
  int eq = 0, gt = 0;
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int i = tg * KPT + q;
    if (i < n) { eq += key[q] == T; gt += key[q] > T; }
  }
  if (eq_total == need_eq) {   // every key equal to T is taken (the usual case): one scan
    int pos = group_excl_scan<GROUP>(gt + eq, S.red[1], bar_id);
#pragma unroll
    for (int q = 0; q < KPT; ++q) {
      const int i = tg * KPT + q;
      if (i < n && key[q] >= T) out[pos++] = base_idx + i;
    }
    if (tg == 0) *cnt_out = k;
    return;
  }
  const int eq_before = group_excl_scan<GROUP>(eq, S.red[0], bar_id);
  const int take = gt + max(0, min(eq, need_eq - eq_before));
  int pos = group_excl_scan<GROUP>(take, S.red[1], bar_id);
  int r = eq_before;
#pragma unroll
  for (int q = 0; q < KPT; ++q) {
    const int i = tg * KPT + q;
    if (i < n) {
      bool t = key[q] > T;
      if (key[q] == T) { t = r < need_eq; ++r; }
      if (t) out[pos++] = base_idx + i;
    }
  }
  if (tg == 0) *cnt_out = k;
}

}  // namespace sa
