// Steps a4 + a5 + a6: paged-gather split-K decode attention over the dense set
// I (sinks + recent window) and each head's selected set J_h, merged exactly
// with the log-sum-exp identity.
//
// HGCA (review, "What carries the argument") attends a recent window densely
// and selected older entries sparsely and fuses the two partial outputs with
//   O = (e^lse_I O_I + e^lse_J O_J) / (e^lse_I + e^lse_J).
// The identity holds for any partition, so here the attended rows of one KV
// head are cut into chunks of whole pages, each chunk keeps a running
// (max, sum, O) per query head, and the last chunk to finish merges all
// chunk partials with the same identity (stabilised by the maximum, as the
// review's comment on Sec. 3.3 asks).
//
// Kernel 1 (tile builder, one CTA per (sequence, KV head)): the union over
// the G query heads of the pages to read, as an ascending list of tiles; a
// tile is one 16-token page with a G-bit head mask per token, so the rows a
// GQA group shares are read once (SPIN abstract / Fig. 6: paged KV substrate).
//
// Kernel 2 (decode, persistent): work items are (KV head unit, chunk of up to
// kTPC tiles).  Lanes of warp 0 look up the page table and issue 2-D TMA
// loads (SWIZZLE_128B, 2 boxes of 16 x 64 bf16 per 4 KB page slab of K and of
// V) completing on one mbarrier per tile.  Each warp then takes whole tiles:
// S = K Q^T and O^T += V^T P on mma.sync m16n8k16 (tokens x heads, heads
// padded to 8), with P split into a bf16 high part and a bf16 residual so the
// product keeps ~16 mantissa bits.
#include <cuda.h>

#include <algorithm>

#include "sa_common.cuh"

namespace sa {

struct __align__(16) Tile {
  int lp;            // logical page
  int pad[3];
  uint32_t mask[4];  // byte i = G-bit mask of heads attending token 16 lp + i
};

constexpr int kBuildThreads = 512;
constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kTPC = 8;                      // tiles per chunk
constexpr int kSlab = kP * kD * 2;           // 4096 bytes: one page of one KV head
constexpr int kTileBytes = 2 * kSlab;        // K + V
constexpr int kBoxBytes = 16 * 64 * 2;       // one TMA box: 16 rows x 64 bf16

// ------------------------------------------------------------------ tile builder

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

__global__ void __launch_bounds__(kBuildThreads)
build_tiles_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ sel_idx,
                   const int* __restrict__ sel_cnt, int gran, Tile* __restrict__ tiles,
                   int* __restrict__ ntiles) {
  extern __shared__ int flag[];  // [mpp]: page flag, then tile index
  __shared__ int scan_tmp[32];
  const int kvh = blockIdx.x, b = blockIdx.y;
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
    if (flag[i]) {
      // dense-set tokens of this page attend for every head
      Tile t;
      t.lp = i;
      t.pad[0] = t.pad[1] = t.pad[2] = 0;
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
      T[base] = t;
      flag[i] = base++;
    } else {
      flag[i] = -1;
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
}

// ------------------------------------------------------------------ decode

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int* page_table;
  const Tile* tiles;
  const int* ntiles;
  float* partials;   // [U][chunk_cap][G][kD + 2]
  int* counters;     // [U]
  float* out;
  float* lse;
  float* logits;     // may be null
  int* status;
  int chunk_cap;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..15) of row `row` inside a K or V
  // slab written by two SWIZZLE_128B boxes of 16 rows x 128 bytes
  return (uint32_t)((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ int nchunks_of(int nt) { return nt > 0 ? (nt + kTPC - 1) / kTPC : 1; }

__global__ void __launch_bounds__(kDecThreads)
decode_kernel(Params p, DecodeArgs A, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base for the swizzled TMA boxes
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_tiles = smem;                                          // kTPC * kTileBytes
  uint8_t* s_p = s_tiles + kTPC * kTileBytes;                       // kDecWarps * 512 bytes
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_p + kDecWarps * 512);   // kTPC
  int* s_phys = reinterpret_cast<int*>(s_bar + kTPC);                // kTPC
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_phys + kTPC);     // kTPC * 4
  int* s_lp = reinterpret_cast<int*>(s_mask + 4 * kTPC);             // kTPC
  int* s_misc = s_lp + kTPC;                                         // [0] last flag, [1] abort
  int* s_prefix = s_misc + 4;                                        // [U + 1]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G;
  const int U = p.B * p.Hk;

  if (tid == 0) {
    for (int i = 0; i < kTPC; ++i) mbar_init(&s_bar[i], 1);
    fence_mbar_init();
    s_misc[1] = 0;
  }
  // work prefix over units: chunks per unit
  for (int i = tid; i < U; i += blockDim.x) s_prefix[i + 1] = nchunks_of(A.ntiles[i]);
  __syncthreads();
  if (tid == 0) {
    s_prefix[0] = 0;
    for (int i = 0; i < U; ++i) s_prefix[i + 1] += s_prefix[i];
  }
  __syncthreads();
  const int total = s_prefix[U];
  uint32_t phase = 0;   // bit i = parity of the next phase of barrier i
  const float scale_log2 = p.scale * 1.4426950408889634f;
  const int g4 = lane >> 2, t4 = lane & 3;

  for (int w = blockIdx.x; w < total; w += gridDim.x) {
    // locate the unit: s_prefix[lo] <= w < s_prefix[lo + 1]
    int lo = 0, hi = U;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_prefix[mid] <= w) lo = mid; else hi = mid;
    }
    const int u = lo;
    const int c = w - s_prefix[u];
    const int nch = s_prefix[u + 1] - s_prefix[u];
    const int b = u / p.Hk, kvh = u % p.Hk;
    const int nt = A.ntiles[u];
    const int t_begin = c * kTPC;
    const int t_cnt = max(0, min(kTPC, nt - t_begin));

    // ---- producer: warp 0 lanes look up pages and issue the TMA loads
    if (warp == 0 && lane < t_cnt) {
      const Tile* tp = A.tiles + (size_t)u * p.mpp + t_begin + lane;
      const int4 w0 = *reinterpret_cast<const int4*>(tp);
      const uint4 w1 = *reinterpret_cast<const uint4*>(&tp->mask[0]);
      const int lp = w0.x;
      const int phys = (lp >= 0 && lp < p.mpp) ? A.page_table[(size_t)b * p.mpp + lp] : -1;
      const bool ok = phys >= 0 && phys < p.num_pages;
      if (!ok) set_status(A.status, SA_ERR_BAD_PAGE);
      s_phys[lane] = ok ? phys : -1;
      s_lp[lane] = lp;
      s_mask[4 * lane + 0] = w1.x; s_mask[4 * lane + 1] = w1.y;
      s_mask[4 * lane + 2] = w1.z; s_mask[4 * lane + 3] = w1.w;
      if (ok) {
        uint8_t* dst = s_tiles + lane * kTileBytes;
        const int row = (phys * p.Hk + kvh) * kP;
        mbar_arrive_expect_tx(&s_bar[lane], kTileBytes);
        tma_load_2d(dst, &tmK, 0, row, &s_bar[lane]);
        tma_load_2d(dst + kBoxBytes, &tmK, 64, row, &s_bar[lane]);
        tma_load_2d(dst + kSlab, &tmV, 0, row, &s_bar[lane]);
        tma_load_2d(dst + kSlab + kBoxBytes, &tmV, 64, row, &s_bar[lane]);
      }
    }
    // Q fragments (B operand: k = dim, n = head), heads >= G are zero
    uint32_t qb[8][2];
    {
      const bool hv = g4 < G;
      const uint32_t* qrow =
          reinterpret_cast<const uint32_t*>(A.q + ((size_t)b * p.Hq + kvh * G + (hv ? g4 : 0)) * kD);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qb[ks][0] = hv ? __ldg(qrow + ks * 8 + t4) : 0u;
        qb[ks][1] = hv ? __ldg(qrow + ks * 8 + 4 + t4) : 0u;
      }
    }
    __syncthreads();

    // ---- consumers: each warp takes whole tiles
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    uint8_t* sp = s_p + warp * 512;
    const uint32_t sp_hi = smem_u32(sp), sp_lo = sp_hi + 256;

    for (int i = warp; i < t_cnt; i += kDecWarps) {
      if (s_phys[i] < 0) continue;
      if (!mbar_wait_bounded(&s_bar[i], (phase >> i) & 1u, A.status)) {
        s_misc[1] = 1;
        continue;
      }
      const uint32_t sK = smem_u32(s_tiles + i * kTileBytes);
      const uint32_t sV = sK + kSlab;
      // S = K Q^T  (rows = tokens, cols = heads)
      float s[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int mi = lane >> 3, r = lane & 7;
        const int row = (mi & 1) * 8 + r;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(sK + swz(row, ks * 2 + (mi >> 1)), a0, a1, a2, a3);
          mma_bf16_16816(s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
      }
      // masks: tokens g4 and g4 + 8, heads 2 t4 and 2 t4 + 1
      const uint32_t mb0 = (s_mask[4 * i + (g4 >> 2)] >> (8 * (g4 & 3))) & 0xffu;
      const uint32_t mb1 = (s_mask[4 * i + 2 + (g4 >> 2)] >> (8 * (g4 & 3))) & 0xffu;
      const int h0 = 2 * t4, h1 = 2 * t4 + 1;
      const bool v00 = (mb0 >> h0) & 1u, v01 = (mb0 >> h1) & 1u;
      const bool v10 = (mb1 >> h0) & 1u, v11 = (mb1 >> h1) & 1u;
      const float z00 = v00 ? s[0] * scale_log2 : -INFINITY;
      const float z01 = v01 ? s[1] * scale_log2 : -INFINITY;
      const float z10 = v10 ? s[2] * scale_log2 : -INFINITY;
      const float z11 = v11 ? s[3] * scale_log2 : -INFINITY;
      float t0 = fmaxf(z00, z10), t1 = fmaxf(z01, z11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
      }
      const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
      const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
      const float al0 = exp2f(m0 - u0), al1 = exp2f(m1 - u1);
      const float p00 = exp2f(z00 - u0), p01 = exp2f(z01 - u1);
      const float p10 = exp2f(z10 - u0), p11 = exp2f(z11 - u1);
      l0 = l0 * al0 + p00 + p10;
      l1 = l1 * al1 + p01 + p11;
      m0 = n0;
      m1 = n1;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
      }
      if (A.logits != nullptr) {
        const int base_tok = s_lp[i] * kP;
        const size_t hs = (size_t)p.mpp * kP;
        const size_t row0 = ((size_t)b * p.Hq + kvh * G) * hs;
        if (v00) A.logits[row0 + h0 * hs + base_tok + g4] = s[0] * p.scale;
        if (v01) A.logits[row0 + h1 * hs + base_tok + g4] = s[1] * p.scale;
        if (v10) A.logits[row0 + h0 * hs + base_tok + g4 + 8] = s[2] * p.scale;
        if (v11) A.logits[row0 + h1 * hs + base_tok + g4 + 8] = s[3] * p.scale;
      }
      // P (tokens x heads) as bf16 high part + bf16 residual
      {
        const __nv_bfloat162 hA = __floats2bfloat162_rn(p00, p01);
        const __nv_bfloat162 hB = __floats2bfloat162_rn(p10, p11);
        const float2 fA = __bfloat1622float2(hA), fB = __bfloat1622float2(hB);
        uint32_t* ph = reinterpret_cast<uint32_t*>(sp);
        uint32_t* pl = reinterpret_cast<uint32_t*>(sp + 256);
        ph[g4 * 4 + t4] = *reinterpret_cast<const uint32_t*>(&hA);
        ph[(g4 + 8) * 4 + t4] = *reinterpret_cast<const uint32_t*>(&hB);
        pl[g4 * 4 + t4] = pack_bf16(p00 - fA.x, p01 - fA.y);
        pl[(g4 + 8) * 4 + t4] = pack_bf16(p10 - fB.x, p11 - fB.y);
      }
      __syncwarp();
      uint32_t bh0, bh1, bl0, bl1;
      ldsm_x2_t(sp_hi + (lane & 15) * 16, bh0, bh1);
      ldsm_x2_t(sp_lo + (lane & 15) * 16, bl0, bl1);
      {
        const int mi = lane >> 3, r = lane & 7;
        const int tok = (mi >> 1) * 8 + r;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(sV + swz(tok, mt * 2 + (mi & 1)), a0, a1, a2, a3);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, bh0, bh1);
          mma_bf16_16816(o[mt], a0, a1, a2, a3, bl0, bl1);
        }
      }
      __syncwarp();
    }
    // row sums over the 8 lanes that share t4
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // flip the phase of every barrier that completed in this chunk
    for (int i = 0; i < t_cnt; ++i)
      if (s_phys[i] >= 0) phase ^= 1u << i;
    __syncthreads();   // all warps done with the tiles; reuse tile smem

    // ---- merge the warps' states: wm/wl [kDecWarps][8], wo [kDecWarps][8][kD]
    float* wm = reinterpret_cast<float*>(s_tiles);
    float* wl = wm + kDecWarps * 8;
    float* wo = wl + kDecWarps * 8;
    if (g4 == 0) {
      wm[warp * 8 + 2 * t4] = m0; wm[warp * 8 + 2 * t4 + 1] = m1;
      wl[warp * 8 + 2 * t4] = l0; wl[warp * 8 + 2 * t4 + 1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int d = mt * 16 + g4;
      wo[(warp * 8 + 2 * t4) * kD + d] = o[mt][0];
      wo[(warp * 8 + 2 * t4 + 1) * kD + d] = o[mt][1];
      wo[(warp * 8 + 2 * t4) * kD + d + 8] = o[mt][2];
      wo[(warp * 8 + 2 * t4 + 1) * kD + d + 8] = o[mt][3];
    }
    __syncthreads();
    const int d = tid;   // kDecThreads == kD
    float* part = A.partials + ((size_t)u * A.chunk_cap + c) * G * (kD + 2);
    for (int g = 0; g < G; ++g) {
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kDecWarps; ++ww) M = fmaxf(M, wm[ww * 8 + g]);
      float acc = 0.f, l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int ww = 0; ww < kDecWarps; ++ww) {
          const float mw = wm[ww * 8 + g];
          const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
          acc += f * wo[(ww * 8 + g) * kD + d];
          l += f * wl[ww * 8 + g];
        }
      }
      if (nch == 1) {
        const size_t row = (size_t)b * p.Hq + kvh * G + g;
        A.out[row * kD + d] = l > 0.f ? acc / l : 0.f;
        if (d == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
      } else {
        part[g * (kD + 2) + d] = acc;
        if (d == 0) {
          part[g * (kD + 2) + kD] = M;
          part[g * (kD + 2) + kD + 1] = l;
        }
      }
    }
    if (nch > 1) {
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int prev = atomicAdd(&A.counters[u], 1);
        s_misc[0] = (prev == nch - 1);
      }
      __syncthreads();
      if (s_misc[0]) {
        __threadfence();
        const float* pu = A.partials + (size_t)u * A.chunk_cap * G * (kD + 2);
        for (int g = 0; g < G; ++g) {
          float M = -INFINITY;
          for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(pu + ((size_t)cc * G + g) * (kD + 2) + kD));
          float acc = 0.f, l = 0.f;
          if (M != -INFINITY) {
            for (int cc = 0; cc < nch; ++cc) {
              const float* pc = pu + ((size_t)cc * G + g) * (kD + 2);
              const float mc = __ldcg(pc + kD);
              const float f = mc == -INFINITY ? 0.f : exp2f(mc - M);
              acc += f * __ldcg(pc + d);
              l += f * __ldcg(pc + kD + 1);
            }
          }
          const size_t row = (size_t)b * p.Hq + kvh * G + g;
          A.out[row * kD + d] = l > 0.f ? acc / l : 0.f;
          if (d == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
        }
        if (tid == 0) A.counters[u] = 0;
      }
    }
    fence_proxy_async_smem();   // generic smem writes above precede the next chunk's TMA writes
    __syncthreads();
    if (s_misc[1]) break;       // a wait ran out: stop taking work
  }
  // a wait that ran out may leave copies in flight: give them a bounded
  // chance to land before the CTA's shared memory is released
  if (s_misc[1] && tid < kTPC) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
      if (mbar_try_wait(&s_bar[tid], (phase >> tid) & 1u)) break;
  }
}

size_t decode_smem_bytes(int U) {
  return 1024 + (size_t)kTPC * kTileBytes + kDecWarps * 512 + kTPC * 8 + kTPC * 4 + kTPC * 16 + kTPC * 4 + 16 +
         (size_t)(U + 1) * 4;
}

int chunk_cap_of(const Params& p) { return (p.mpp + kTPC - 1) / kTPC; }

size_t tiles_bytes(const Params& p) { return (size_t)p.B * p.Hk * p.mpp * sizeof(Tile); }

int launch_build_tiles(const Params& p, const int* seq_lens, const int* sel_idx, const int* sel_cnt, int gran,
                       void* tiles, int* ntiles, cudaStream_t stream) {
  const size_t smem = (size_t)p.mpp * sizeof(int);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(p.Hk, p.B);
  build_tiles_kernel<<<grid, kBuildThreads, smem, stream>>>(p, seq_lens, sel_idx, sel_cnt, gran,
                                                            static_cast<Tile*>(tiles), ntiles);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int launch_decode(const Params& p, const void* q, const int* page_table, const void* tiles, const int* ntiles,
                  float* partials, int* counters, float* out, float* lse, float* logits, int* status,
                  const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  const int U = p.B * p.Hk;
  const size_t smem = decode_smem_bytes(U);
  if (smem > 227 * 1024) return SA_ERR_UNSUPPORTED;
  cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel, kDecThreads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int chunk_cap = chunk_cap_of(p);
  const long long max_work = (long long)U * chunk_cap;
  const int grid = (int)std::min<long long>(max_work, (long long)num_sms * per_sm);
  DecodeArgs A;
  A.q = static_cast<const __nv_bfloat16*>(q);
  A.page_table = page_table;
  A.tiles = static_cast<const Tile*>(tiles);
  A.ntiles = ntiles;
  A.partials = partials;
  A.counters = counters;
  A.out = out;
  A.lse = lse;
  A.logits = logits;
  A.status = status;
  A.chunk_cap = chunk_cap;
  decode_kernel<<<grid, kDecThreads, smem, stream>>>(p, A, tmK, tmV);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
