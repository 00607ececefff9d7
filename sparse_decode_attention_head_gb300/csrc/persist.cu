// One decode step in one persistent launch: block scores (a2), per-head
// top-k (a3), tile lists (a4/a5 set-up), paged decode (a4 + a5) and the exact
// log-sum-exp merge (a6), with the tail-block summary refresh (a1).
//
// The step's phases depend on each other per (sequence, KV head) unit only:
// a unit's top-k needs that unit's scores, its decode needs its top-k.  So
// instead of one kernel per phase (each paying its start-up latency while the
// previous drains), the phases are work queues between warp roles of one
// persistent grid, one CTA per SM:
//   - 8 consumer warps stream.  First score items: a run of one unit's block
//     summaries plus the group's q, copied into a warp-owned 8 KB shared
//     memory slot by one bulk copy; the warp scores the run for every head of
//     the group in the canonical fp32 order and adds the run's blocks to the
//     unit's scored count.  Items are claimed from a global ticket in
//     unit-major order, so units finish scoring one after another.  Then
//     decode tiles: each KV page of a chunk (K and V, 8 KB) lands in a slot by
//     two TMA copies; the warp runs S = K Q^T and O^T += V^T P on mma.sync.
//     Each warp issues its own copies (2 or 3 slots in flight), so no
//     producer hand-off sits between a freed slot and its next copy.
//   - 4 selector warps take (unit, head) tickets: once the unit is scored they
//     run the head's top-k (radix select over the scores in L2); the last head
//     of a unit builds its tile list (page bitmaps, head masks per token),
//     refreshes the tail summary and publishes the unit's chunks in a global
//     queue.  HGCA (review, "What carries the argument") splits attention into
//     a dense part over the newest entries and a sparse part over selected
//     older ones; Fluxion (core claim, Fig. 2) selects blocks per head.
//   - 1 control warp takes chunk tickets from the queue (one ahead), stages
//     the chunk's tile descriptors and q in a shared-memory ring, and
//     publishes it to the consumers.
// A chunk's tiles are split among the 8 consumer warps; each parks its
// online-softmax state, the last one combines the 8 states into the chunk's
// partial; the last chunk of a unit merges the unit's partials with the
// identity O = sum_c e^{m_c - M} O_c / sum_c e^{m_c - M} l_c (HGCA, the fusion
// of partial attentions, applied to a chain; stabilised by the maximum).
//
// All work is claimed from global tickets, so the launch completes whichever
// CTAs are resident; every wait is bounded and records SA_ERR_TIMEOUT.  The
// last CTA to leave zeroes the launch's counters for the next launch.
#include <cuda.h>

#include <algorithm>

#include "persist.cuh"
#include "score_core.cuh"
#include "summary.cuh"
#include "topk.cuh"

namespace sa {

namespace {

constexpr int kPSel = 4;                         // selector warps (warps 0..3)
constexpr int kPC = 8;                           // consumer warps (warps 4..11)
constexpr int kPCtl = kPSel + kPC;               // the control warp (warp 12)
constexpr int kPThreads = (kPSel + kPC + 1) * 32;
constexpr int kSelThreads = kPSel * 32;
constexpr int kSlotB = 8192;                     // one K + V page of a KV head, or one score item
constexpr int kSlab = kP * kD * 2;               // 4096 bytes: one page of K (or V)
constexpr int kBoxB = 16 * 64 * 2;               // one TMA box: 16 rows x 64 bf16
constexpr int kPRing = 3;                        // chunk ring entries
constexpr int kFifo = 8;                         // per-warp issued-entry ring (slots + park markers)
constexpr int kQOff = 6144;                      // score item: q rows at this offset of the slot
constexpr int kItemBatch = 2;                    // score items a warp claims per ticket (one atomic)
constexpr int kPartF = kD + 2;                   // floats per head in a parked state: O, max, sum
constexpr int kBuildWin = 1024;                  // pages per tile-builder window
constexpr int kHbWords = 64;                     // block-bitmap words per head and window (2048 blocks)
constexpr uint32_t kSpin = 1u << 22;             // bounded waits on shared memory (polls)
constexpr uint32_t kSpinGlobal = 1u << 20;       // bounded waits on global memory (polls, each an L2 round trip)

enum { kScore = 1, kTile = 2, kPark = 3 };

// score item: summary rows of one unit (6 KB) then the group's q
__host__ __device__ constexpr int item_rows(int mode) { return mode == SA_SUMMARY_MINMAX ? 12 : 24; }

struct RingHdr {   // one published chunk
  int unit, t0, nt, nch, pos0, kin, pad[2];
};

// misc ints in shared memory
enum { M_PUB = 0, M_COMB, M_PARKED, M_SEL_T, M_SEL_OK, M_SEL_LAST, M_LASTCTA, M_QTAIL, M_SCAN = 8, M_NMISC = 16 };

struct Smem {
  uint8_t* slots;
  int* items;        // [U + 1] score items before unit u
  uint8_t* ring_q;   // [kPRing][G * kD] bf16
  Tile* ring_tiles;  // [kPRing][kPMaxC]
  float* park;       // [kPC][G][kPartF]
  uint8_t* pbuf;     // [kPC][512] P tiles
  RingHdr* hdr;      // [kPRing]
  int4* fifo;        // [kPC][kFifo]
  uint64_t* full;    // [kPC][3]
  int* misc;         // [M_NMISC]
  TopkScratch* topk;
  uint32_t* hb;      // [kMaxG][kHbWords] head block bitmaps
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

// Byte offsets of the shared-memory regions (base aligned to 1024).
struct SmemPlan {
  size_t slots, items, ring_q, ring_tiles, park, pbuf, hdr, fifo, full, misc, topk, hb, total;
};

__host__ __device__ inline SmemPlan smem_plan(int U, int G, int nslots) {
  SmemPlan s;
  size_t o = 0;
  s.slots = o;      o += (size_t)kPC * nslots * kSlotB;
  s.items = o;      o = align16(o + (size_t)(U + 1) * 4);
  s.ring_q = o;     o += (size_t)kPRing * G * kD * 2;
  s.ring_tiles = o; o += (size_t)kPRing * kPMaxC * sizeof(Tile);
  s.park = o;       o += (size_t)kPC * G * kPartF * 4;
  s.pbuf = o;       o += (size_t)kPC * 512;
  s.hdr = o;        o += (size_t)kPRing * sizeof(RingHdr);
  s.fifo = o;       o += (size_t)kPC * kFifo * sizeof(int4);
  s.full = o;       o += (size_t)kPC * 3 * 8;
  s.misc = o;       o += M_NMISC * 4;
  s.topk = o;       o = align16(o + sizeof(TopkScratch));
  s.hb = o;         o += (size_t)kMaxG * kHbWords * 4;
  s.total = o + 1024;   // room to align the base
  return s;
}

__device__ __forceinline__ void sel_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSelThreads) : "memory"); }

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..15) of row `row` inside a K or V
  // slab written by two SWIZZLE_128B boxes of 16 rows x 128 bytes
  return (uint32_t)((chunk >> 3) * kBoxB + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Unit u with prefix[u] <= x < prefix[u + 1].
__device__ __forceinline__ int unit_of_item(const int* prefix, int U, int x) {
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// bits 0, 8, 16, 24 set from the four bits of n
__device__ __forceinline__ uint32_t spread4(uint32_t n) {
  return (n & 1u) | ((n & 2u) << 7) | ((n & 4u) << 14) | ((n & 8u) << 21);
}

// Bounded poll (one lane) until *x >= v: relaxed loads, then one acquire
// fence once the value is seen.  False on timeout.
__device__ __forceinline__ bool wait_ge_gpu(const int* x, int v) {
  for (uint32_t i = 0; i < kSpinGlobal; ++i) {
    if (ld_relaxed_gpu(x) >= v) {
      fence_acq_rel_gpu();
      return true;
    }
    __nanosleep(64);
  }
  return false;
}

// ------------------------------------------------------------------ consumer: score one item

template <int MODE>
__device__ __forceinline__ void score_item(const Params& p, const PArgs& A, const uint8_t* stage, int u, int first,
                                           int nb, int lane) {
  constexpr int kRowB = (MODE == SA_SUMMARY_MINMAX ? 2 : 1) * kD * 2;
  constexpr int kRows = item_rows(MODE);
  const int G = p.G;
  const int b = u / p.Hk, kvh = u % p.Hk;
  const int L = min(__ldg(A.seq_lens + b), p.mpp * kP);
  int j0, j1;
  candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
  const int sub = lane >> 3, part = lane & 7;
  const long long sbase = ((long long)b * p.Hq + kvh * G) * p.slots + j0 + first;
  for (int hs = 0; hs * 4 < G; ++hs) {
    QSet4 qs;
    qset_load(qs, stage + kQOff, hs, G, part);
#pragma unroll
    for (int r = 0; r < kRows / 4; ++r) {
      const int cl = r * 4 + sub;
      const bool valid = cl < nb;
      float acc[4];
      dot4_part<MODE>(qs, stage + (size_t)(valid ? cl : 0) * kRowB, part, acc);
      const float v = butterfly4(acc, part);
      const int g = hs * 4 + (part >> 1);
      if (valid && (part & 1) == 0 && g < G) A.scores[sbase + (long long)g * p.slots + cl] = v;
    }
  }
}

// ------------------------------------------------------------------ consumer: one decode tile

struct AttnState {
  float m0, m1, l0, l1;
  float o[8][4];
};

__device__ __forceinline__ void attn_reset(AttnState& s) {
  s.m0 = s.m1 = -INFINITY;
  s.l0 = s.l1 = 0.f;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) s.o[mt][0] = s.o[mt][1] = s.o[mt][2] = s.o[mt][3] = 0.f;
}

// S = K Q^T (tokens x heads) and O^T += V^T P for one 16-token page; masks:
// byte i of the 16 bytes = the heads attending token i.  P goes through the
// warp's 512-byte buffer as a bf16 high part and a bf16 residual.
__device__ __forceinline__ void attend_tile(const uint8_t* slot, const Tile& t, const uint32_t (&qb)[8][2],
                                            float scale_log2, AttnState& s, uint8_t* sp, int lane) {
  const int g4 = lane >> 2, t4 = lane & 3;
  const uint32_t sK = smem_u32(slot), sV = sK + kSlab;
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
  {
    const int mi = lane >> 3, r = lane & 7;
    const int row = (mi & 1) * 8 + r;
#pragma unroll
    for (int ks = 0; ks < 8; ks += 2) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(sK + swz(row, ks * 2 + (mi >> 1)), a0, a1, a2, a3);
      mma_bf16_16816(sa, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      ldsm_x4(sK + swz(row, (ks + 1) * 2 + (mi >> 1)), a0, a1, a2, a3);
      mma_bf16_16816(sb, a0, a1, a2, a3, qb[ks + 1][0], qb[ks + 1][1]);
    }
  }
  const float s0 = sa[0] + sb[0], s1 = sa[1] + sb[1], s2 = sa[2] + sb[2], s3 = sa[3] + sb[3];
  // tokens g4 and g4 + 8, heads 2 t4 and 2 t4 + 1
  const uint32_t mb0 = (t.mask[g4 >> 2] >> (8 * (g4 & 3))) & 0xffu;
  const uint32_t mb1 = (t.mask[2 + (g4 >> 2)] >> (8 * (g4 & 3))) & 0xffu;
  const int h0 = 2 * t4, h1 = 2 * t4 + 1;
  const bool v00 = (mb0 >> h0) & 1u, v01 = (mb0 >> h1) & 1u;
  const bool v10 = (mb1 >> h0) & 1u, v11 = (mb1 >> h1) & 1u;
  const float z00 = v00 ? s0 * scale_log2 : -INFINITY;
  const float z01 = v01 ? s1 * scale_log2 : -INFINITY;
  const float z10 = v10 ? s2 * scale_log2 : -INFINITY;
  const float z11 = v11 ? s3 * scale_log2 : -INFINITY;
  float t0 = fmaxf(z00, z10), t1 = fmaxf(z01, z11);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
    t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
  }
  const float n0 = fmaxf(s.m0, t0), n1 = fmaxf(s.m1, t1);
  const float u0 = n0 == -INFINITY ? 0.f : n0, u1 = n1 == -INFINITY ? 0.f : n1;
  const float al0 = exp2f(s.m0 - u0), al1 = exp2f(s.m1 - u1);
  const float p00 = exp2f(z00 - u0), p01 = exp2f(z01 - u1);
  const float p10 = exp2f(z10 - u0), p11 = exp2f(z11 - u1);
  s.l0 = s.l0 * al0 + p00 + p10;
  s.l1 = s.l1 * al1 + p01 + p11;
  s.m0 = n0;
  s.m1 = n1;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    s.o[mt][0] *= al0; s.o[mt][1] *= al1; s.o[mt][2] *= al0; s.o[mt][3] *= al1;
  }
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
  const uint32_t sp_hi = smem_u32(sp), sp_lo = sp_hi + 256;
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
      mma_bf16_16816(s.o[mt], a0, a1, a2, a3, bh0, bh1);
      mma_bf16_16816(s.o[mt], a0, a1, a2, a3, bl0, bl1);
    }
  }
}

// ------------------------------------------------------------------ merge of a unit's chunk partials

// The 128 selector threads: the exact merge of the nch partials of unit u
// (HGCA's fusion identity over a chain, stabilised by the maximum).  Warp w
// merges heads w, w + 4; lane j holds chunk j's (max, sum) (32 chunks at a
// time), the weights e^{m_j - M} go round by shuffles, and the O rows (lane
// owns dims [4 lane, 4 lane + 4)) are loaded eight chunks at a time, so the
// L2 round trips overlap.
__device__ void merge_unit(const Params& p, const PArgs& A, int u, int pos0, int nch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int G = p.G, PS = partial_stride(G);
  const float* P = A.partials + (size_t)pos0 * PS;
  const int b = u / p.Hk, kvh = u % p.Hk;
  for (int g = w; g < G; g += kPSel) {
    float M = -INFINITY;
    for (int j = lane; j < nch; j += 32) M = fmaxf(M, __ldcg(P + (size_t)j * PS + G * kD + g));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (M != -INFINITY) {
      for (int j0 = 0; j0 < nch; j0 += 32) {
        const int j = j0 + lane;
        float mj = -INFINITY, lj = 0.f;
        if (j < nch) {
          mj = __ldcg(P + (size_t)j * PS + G * kD + g);
          lj = __ldcg(P + (size_t)j * PS + G * kD + G + g);
        }
        const float fj = mj == -INFINITY ? 0.f : exp2f(mj - M);
        float lw = fj * lj;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, off);
        l += lw;
        const int nb = min(32, nch - j0);
        for (int c0 = 0; c0 < nb; c0 += 8) {
          float4 x[8];
#pragma unroll
          for (int c = 0; c < 8; ++c)
            x[c] = c0 + c < nb ? __ldcg(reinterpret_cast<const float4*>(P + (size_t)(j0 + c0 + c) * PS + g * kD) + lane)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float f = __shfl_sync(0xffffffffu, fj, (c0 + c) & 31);
            acc.x += f * x[c].x;
            acc.y += f * x[c].y;
            acc.z += f * x[c].z;
            acc.w += f * x[c].w;
          }
        }
      }
    }
    const size_t row = (size_t)b * p.Hq + kvh * G + g;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    reinterpret_cast<float4*>(A.out + row * kD)[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (lane == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
  }
}

// ------------------------------------------------------------------ selector: tile list of a unit

// The 128 selector threads: tiles of unit u from the G heads' selections (block
// ids, global memory), in windows of kBuildWin pages.  Per window: a bit per
// selected block per head; then per 32-page word the pages to read (pages
// with dense-set tokens, and pages of selected blocks -- every such page holds
// a token of M or of the dense set); a prefix of their counts; and one
// 32-byte descriptor per touched page with its 16 per-token head masks.
// Returns the tile count (valid in every selector thread).
__device__ int build_unit(const Params& p, const PArgs& A, const Smem& S, int u) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int G = p.G;
  const int b = u / p.Hk, kvh = u % p.Hk;
  const int Lc = max(0, min(__ldg(A.seq_lens + b), p.mpp * kP));
  const int npg = (Lc + kP - 1) / kP;
  int s_end, w_beg;
  partition(Lc, p.S, p.W, s_end, w_beg);
  const int Bs = p.bs[kvh];
  const int lgB = Bs == 8 ? 3 : Bs == 16 ? 4 : Bs == 32 ? 5 : 6;
  const uint32_t all = (1u << G) - 1u;
  const size_t h0 = (size_t)b * p.Hq + kvh * G;
  const int* sel_row = A.sel_idx + h0 * p.kcap;
  const int* cnt_row = A.sel_cnt + h0;
  const int* pt_row = A.page_table + (size_t)b * p.mpp;
  Tile* T = A.tiles + (size_t)u * p.mpp;
  uint32_t* touched = S.topk->cand;                             // [32] page words of the window
  int* wpre = S.topk->hist;                                     // [33] tiles before word w; [32] = window total
  // pages holding dense-set tokens: [0, ceil(s_end / P)) and [w_beg / P, npg)
  const int d_lo_end = (s_end + kP - 1) / kP, d_hi_beg = w_beg / kP;
  int* cnt_s = wpre + 40;   // [G] the heads' list lengths (hist[40 ..])
  if (tid < G) cnt_s[tid] = max(0, min(__ldcg(cnt_row + tid), p.kcap));
  sel_sync();
  int total = 0;
  for (int p0 = 0; p0 < npg; p0 += kBuildWin) {
    const int pw = min(kBuildWin, npg - p0);
    const int blk0 = (p0 * kP) >> lgB;                        // first block of the window
    const int nbw = ((pw * kP) + Bs - 1) >> lgB;              // blocks touching the window (<= 2048)
    for (int i = tid; i < G * kHbWords; i += kSelThreads) S.hb[i] = 0u;
    sel_sync();
    for (int it0 = 0; it0 < G * p.kcap; it0 += 4 * kSelThreads) {   // four list entries in flight a thread
      int xv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int it = it0 + r * kSelThreads + tid;
        const int g = it / p.kcap;
        xv[r] = (it < G * p.kcap && it - g * p.kcap < cnt_s[g]) ? __ldcg(sel_row + it) : -1;
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int it = it0 + r * kSelThreads + tid;
        const int x = xv[r] - blk0;
        if (xv[r] < 0 || x < 0 || x >= nbw) continue;
        atomicOr(&S.hb[(it / p.kcap) * kHbWords + (x >> 5)], 1u << (x & 31));
      }
    }
    sel_sync();
    if (tid < 32) {   // word tid: pages p0 + 32 tid .. + 31
      const int q0 = 32 * tid;
      uint32_t sel = 0u;
      for (int g = 0; g < G; ++g) {
        const uint32_t* hb = S.hb + g * kHbWords;
        if (Bs == 16) {
          sel |= hb[tid];
        } else if (Bs == 8) {   // page x: blocks 2x, 2x + 1
          const uint64_t w2 = ((uint64_t)hb[2 * tid + 1] << 32) | hb[2 * tid];
          uint32_t v = 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) v |= (uint32_t)(((w2 >> (2 * i)) & 3ull) != 0ull) << i;
          sel |= v;
        } else {   // Bs = 32 / 64: page x lies in block x >> (lgB - 4)
          const int sh = lgB - 4;
          const int jb = q0 >> sh;
          const uint32_t bits = hb[jb >> 5] >> (jb & 31);
          uint32_t v = 0u;
#pragma unroll
          for (int i = 0; i < 32; ++i) v |= ((bits >> (i >> sh)) & 1u) << i;
          sel |= v;
        }
      }
      // dense pages of this word
      const int a = p0 + q0;
      auto range_bits = [&](int lo, int hi) -> uint32_t {   // pages [lo, hi) within [a, a + 32)
        lo = max(lo, a) - a;
        hi = min(hi, a + 32) - a;
        if (lo >= hi) return 0u;
        const uint32_t up = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
        return up & ~((1u << lo) - 1u);
      };
      uint32_t t = (sel | range_bits(0, d_lo_end) | range_bits(d_hi_beg, npg)) & range_bits(p0, p0 + pw);
      touched[tid] = t;
      const int c = __popc(t);
      const int incl = warp_incl_scan(c);
      wpre[tid] = incl - c;
      if (tid == 31) wpre[32] = incl;
    }
    sel_sync();
    {   // thread t: word t >> 2, pages 8 (t & 3) .. + 7 of it
      const int wd = tid >> 2, qb = (tid & 3) * 8;
      const uint32_t tw = touched[wd];
      uint32_t mine = (tw >> qb) & 0xffu;
      int idx = total + wpre[wd] + __popc(tw & ((1u << qb) - 1u));
      int ph[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ph[i] = ((mine >> i) & 1u) ? __ldg(pt_row + p0 + 32 * wd + qb + i) : -1;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (!((mine >> i) & 1u)) continue;
        const int x = 32 * wd + qb + i;   // page within the window
        const int lp = p0 + x;
        const int tok0 = lp * kP;
        auto rng = [](int lo, int hi) -> uint32_t {   // token bits [lo, hi) of the page
          lo = min(max(lo, 0), kP);
          hi = min(max(hi, 0), kP);
          return lo < hi ? (((1u << hi) - 1u) & ~((1u << lo) - 1u)) : 0u;
        };
        const uint32_t inM = rng(s_end - tok0, w_beg - tok0);
        const uint32_t dense = rng(0, Lc - tok0) & ~inM;
        uint32_t h_lo = 0u, h_hi = 0u;   // heads selecting rows 0-7 / 8-15 of the page
        if (inM != 0u) {
          for (int g = 0; g < G; ++g) {
            const uint32_t* hb = S.hb + g * kHbWords;
            if (Bs == 8) {
              const int j = 2 * x;
              const uint32_t bits = (hb[j >> 5] >> (j & 31)) & 3u;
              h_lo |= (bits & 1u) << g;
              h_hi |= ((bits >> 1) & 1u) << g;
            } else {
              const int j = (x * kP) >> lgB;
              const uint32_t bit = (hb[j >> 5] >> (j & 31)) & 1u;
              h_lo |= bit << g;
              h_hi |= bit << g;
            }
          }
        }
        uint32_t m[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t hsel = q4 < 2 ? h_lo : h_hi;
          m[q4] = spread4((dense >> (4 * q4)) & 15u) * all | spread4((inM >> (4 * q4)) & 15u) * hsel;
        }
        const bool ok = ph[i] >= 0 && ph[i] < p.num_pages;
        if (!ok) set_status(A.status, SA_ERR_BAD_PAGE);
        int4* dst = reinterpret_cast<int4*>(T + idx);
        dst[0] = make_int4(lp, ok ? ph[i] : -1, 0, 0);
        dst[1] = make_int4((int)m[0], (int)m[1], (int)m[2], (int)m[3]);
        ++idx;
      }
    }
    total += wpre[32];
    sel_sync();   // the window's bitmaps and words are reused
  }
  (void)lane;
  return total;
}

// ------------------------------------------------------------------ consumer: combine a chunk

// The last warp to park chunk k combines the kPC parked states (lane owns
// dims [4 lane, 4 lane + 4)) into the chunk's partial, or into the output for
// a unit held in one chunk, releases the park buffer and the chunk's ring
// entry, and counts the chunk for the unit's merge (done by selector warps).
__device__ __forceinline__ void combine_chunk(const Params& p, const PArgs& A, const Smem& S, int k, int lane,
                                           int* unit_done) {
  const int G = p.G;
  if (lane == 0) S.misc[M_PARKED] = 0;
  const RingHdr* h = S.hdr + k % kPRing;
  const int unit = h->unit, nch = h->nch, pos0 = h->pos0, kin = h->kin;
  const int b = unit / p.Hk, kvh = unit % p.Hk;
  float* part = A.partials + (size_t)(pos0 + kin) * partial_stride(G);
  for (int g = 0; g < G; ++g) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPC; ++w) M = fmaxf(M, S.park[(w * G + g) * kPartF + kD]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kPC; ++w) {
        const float* sw = S.park + (w * G + g) * kPartF;
        const float mw = sw[kD];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        const float2 x0 = *reinterpret_cast<const float2*>(sw + 4 * lane);
        const float2 x1 = *reinterpret_cast<const float2*>(sw + 4 * lane + 2);
        acc.x += f * x0.x;
        acc.y += f * x0.y;
        acc.z += f * x1.x;
        acc.w += f * x1.y;
        l += f * sw[kD + 1];
      }
    }
    if (nch == 1) {
      const size_t row = (size_t)b * p.Hq + kvh * G + g;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      reinterpret_cast<float4*>(A.out + row * kD)[lane] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (lane == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
    } else {
      reinterpret_cast<float4*>(part + g * kD)[lane] = acc;
      if (lane == 0) {
        part[G * kD + g] = M;
        part[G * kD + G + g] = l;
      }
    }
  }
  // the park buffer and the chunk's ring entry are free now (the fields above are in registers)
  __syncwarp();
  if (lane == 0) st_release_block(&S.misc[M_COMB], k + 1);
  if (nch > 1) {   // every lane's partial before lane 0's release of the count the merge waits for
    __syncwarp();
    if (lane == 0) red_release_gpu_add(unit_done + unit, 1);
  }
}

// ------------------------------------------------------------------ the kernel

template <int MODE>
__global__ void __launch_bounds__(kPThreads, 1)
step_kernel(Params p, PArgs A, const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int U = p.B * p.Hk;
  const int G = p.G;
  const int nslots = A.nslots;
  const SmemPlan pl = smem_plan(U, G, nslots);
  Smem S;
  S.slots = base + pl.slots;
  S.items = reinterpret_cast<int*>(base + pl.items);
  S.ring_q = base + pl.ring_q;
  S.ring_tiles = reinterpret_cast<Tile*>(base + pl.ring_tiles);
  S.park = reinterpret_cast<float*>(base + pl.park);
  S.pbuf = base + pl.pbuf;
  S.hdr = reinterpret_cast<RingHdr*>(base + pl.hdr);
  S.fifo = reinterpret_cast<int4*>(base + pl.fifo);
  S.full = reinterpret_cast<uint64_t*>(base + pl.full);
  S.misc = reinterpret_cast<int*>(base + pl.misc);
  S.topk = reinterpret_cast<TopkScratch*>(base + pl.topk);
  S.hb = reinterpret_cast<uint32_t*>(base + pl.hb);
  int* gs = A.gs;
  int* unit_scored = gs + kGsHead;
  int* unit_heads = unit_scored + U;
  int* unit_done = unit_heads + U;
  int* unit_pos0 = unit_done + U;
  int* unit_nch1 = unit_pos0 + U;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int kRows = item_rows(MODE);
  constexpr int kRowB = (MODE == SA_SUMMARY_MINMAX ? 2 : 1) * kD * 2;
  constexpr int kRowE = kRowB / 2;

  // ---- prologue: barriers, the per-unit score-item prefix, shared state
  if (tid == 0) {
    for (int i = 0; i < kPC * nslots; ++i) mbar_init(&S.full[(i / nslots) * 3 + i % nslots], 1);
    fence_mbar_init();
    for (int i = 0; i < M_NMISC; ++i) S.misc[i] = 0;
  }
  for (int u = tid; u < U; u += blockDim.x) {
    int items = 0;
    if (!A.given) {
      const int b = u / p.Hk, kvh = u % p.Hk;
      const int L = min(__ldg(A.seq_lens + b), p.mpp * kP);
      int j0, j1;
      candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
      const int n = j1 - j0;
      bool need = false;
      for (int g = 0; g < G; ++g) need |= p.k[kvh * G + g] > 0 && p.k[kvh * G + g] < n;
      items = need ? (n + kRows - 1) / kRows : 0;
    }
    S.items[u + 1] = items;
  }
  __syncthreads();
  if (warp == 0) {   // inclusive scan of the item counts, 32 units at a time
    int carry = 0;
    for (int b0 = 0; b0 < U; b0 += 32) {
      const int u = b0 + lane;
      const int x = warp_incl_scan(u < U ? S.items[u + 1] : 0);
      if (u < U) S.items[u + 1] = x + carry;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) S.items[0] = 0;
  }
  __syncthreads();
  const int total_items = S.items[U];

  if (warp < kPSel) {
    // ================================================================ selectors
    for (;;) {
      if (tid == 0) S.misc[M_SEL_T] = atomicAdd(&gs[kGsSelTicket], 1);
      sel_sync();
      const int t = S.misc[M_SEL_T];
      sel_sync();
      int u;
      bool build = false;
      if (A.given) {
        if (t >= U) break;
        u = t;
        build = true;
      } else {
        if (t >= U * G) break;
        u = t / G;
        const int g = t - u * G;
        const int b = u / p.Hk, kvh = u % p.Hk, h = kvh * G + g;
        const int L = min(__ldg(A.seq_lens + b), p.mpp * kP);
        int j0, j1;
        candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
        const int n = j1 - j0, k = p.k[h];
        if (k > 0 && k < n) {   // the head ranks scores: wait until the unit is scored
          if (tid == 0) {
            const bool ok = wait_ge_gpu(unit_scored + u, n);
            if (!ok) set_status(A.status, SA_ERR_TIMEOUT);
            S.misc[M_SEL_OK] = ok;
          }
          sel_sync();
          if (!S.misc[M_SEL_OK]) break;   // (the merge loop below then times out too, bounded)
        }
        const float* sc = A.scores + ((size_t)b * p.Hq + h) * p.slots + j0;
        int* out_idx = A.sel_idx + ((size_t)b * p.Hq + h) * p.kcap;
        int* out_cnt = A.sel_cnt + (size_t)b * p.Hq + h;
        if (n <= kSelThreads * 16)
          group_topk<kSelThreads, 16, false, true>(sc, n, k, j0, out_idx, out_cnt, 1, *S.topk);
        else
          group_topk_stream<kSelThreads>(sc, n, k, j0, out_idx, out_cnt, 1, *S.topk);
        sel_sync();   // every thread's list entries before thread 0's release of the count
        if (tid == 0) S.misc[M_SEL_LAST] = atom_acq_rel_gpu_add(unit_heads + u, 1) == G - 1;
        sel_sync();
        build = S.misc[M_SEL_LAST] != 0;
      }
      if (!build) continue;
      // ---- the unit's tile list, its chunks, and (step) the tail summary
      const int total = build_unit(p, A, S, u);
      const int b = u / p.Hk, kvh = u % p.Hk;
      if (total == 0) {   // nothing attended (L = 0): O = 0, lse = -inf
        for (int i = tid; i < G * kD; i += kSelThreads) A.out[((size_t)b * p.Hq + kvh * G) * kD + i] = 0.f;
        if (tid < G) A.lse[(size_t)b * p.Hq + kvh * G + tid] = -INFINITY;
      }
      const int C = max(A.C, (total + kPMaxChunksUnit - 1) / kPMaxChunksUnit);
      const int nch = (total + C - 1) / C;
      sel_sync();   // every thread's tiles before the released queue flags below
      if (tid == 0) S.misc[M_QTAIL] = nch > 0 ? atomicAdd(&gs[kGsQTail], nch) : 0;
      sel_sync();
      const int pos0 = S.misc[M_QTAIL];
      for (int i = tid; i < nch; i += kSelThreads) {
        if (pos0 + i >= A.qcap) {   // cannot happen with the host's sizing; never write past the queue
          set_status(A.status, SA_ERR_CAPACITY);
          continue;
        }
        PQEntry* e = A.dq + pos0 + i;
        e->unit = u;
        e->t0 = i * C;
        e->nt = min(C, total - i * C);
        e->nch = nch;
        e->pos0 = pos0;
        e->kin = i;
        st_release_gpu(&e->flag, 1);
      }
      if (A.summ_w != nullptr && warp == 0) {   // the block holding the newest token, re-summarised
        const int L = min(__ldg(A.seq_lens + b), p.mpp * kP);
        if (L > 0)
          summarize_block_warp(p, b, kvh, (L - 1) / p.bs[kvh], L, A.k_pool, A.page_table + (size_t)b * p.mpp,
                               A.summ_w, A.status);
      }
      sel_sync();
      if (tid == 0) {
        unit_pos0[u] = pos0;
        st_release_gpu(unit_nch1 + u, nch + 1);
        red_release_gpu_add(&gs[kGsUnitsBuilt], 1);
      }
    }
    // ---- then merge tickets: a unit held in several chunks is merged once they are all combined
    for (;;) {
      if (tid == 0) S.misc[M_SEL_T] = atomicAdd(&gs[kGsMergeTicket], 1);
      sel_sync();
      const int u = S.misc[M_SEL_T];
      sel_sync();
      if (u >= U) break;
      if (tid == 0) {
        int nch1 = 0, ok = 1;
        uint32_t i = 0;
        while ((nch1 = ld_relaxed_gpu(unit_nch1 + u)) == 0 && ++i < kSpinGlobal) __nanosleep(64);
        fence_acq_rel_gpu();
        if (nch1 > 2) ok = wait_ge_gpu(unit_done + u, nch1 - 1);
        if (i >= kSpinGlobal || !ok) {
          set_status(A.status, SA_ERR_TIMEOUT);
          nch1 = -1;   // stop: the waits of later tickets would run out too
        }
        S.misc[M_SEL_OK] = nch1;
      }
      sel_sync();
      if (S.misc[M_SEL_OK] < 0) break;
      const int nch = S.misc[M_SEL_OK] - 1;
      if (nch > 1) merge_unit(p, A, u, __ldcg(unit_pos0 + u), nch);
      sel_sync();
    }
  } else if (warp == kPCtl) {
    // ================================================================ control: chunk tickets -> ring
    int tick = 0;
    if (lane == 0) tick = atomicAdd(&gs[kGsQHead], 1);
    for (int k = 0;; ++k) {
      bool ok = true;
      if (lane == 0) {   // ring entry k % kPRing is free once chunk k - kPRing is combined
        uint32_t i = 0;
        while (ld_relaxed_block(&S.misc[M_COMB]) < k - kPRing + 1 && ++i < kSpin) __nanosleep(32);
        ok = i < kSpin;
        fence_acq_rel_block();
      }
      ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
      const int t = __shfl_sync(0xffffffffu, tick, 0);
      if (lane == 0 && ok) tick = atomicAdd(&gs[kGsQHead], 1);
      // wait for queue entry t, or learn that there will be none
      int state = ok ? 0 : 2;   // 0 wait, 1 entry, 2 end / timeout
      if (lane == 0 && ok) {
        for (uint32_t i = 0; i < kSpinGlobal; ++i) {
          if (t < A.qcap && ld_relaxed_gpu(&A.dq[t].flag) != 0) { state = 1; break; }
          if ((i & 7) == 7 && ld_relaxed_gpu(&gs[kGsUnitsBuilt]) >= U) {
            fence_acq_rel_gpu();
            if (t >= ld_relaxed_gpu(&gs[kGsQTail])) {
              state = 2;
              break;
            }
          }
          __nanosleep(32);
        }
        fence_acq_rel_gpu();
        if (state == 0) {
          set_status(A.status, SA_ERR_TIMEOUT);
          state = 2;
        }
      }
      state = __shfl_sync(0xffffffffu, state, 0);
      __syncwarp();   // the entry's fields, ordered after lane 0's acquire of its flag
      RingHdr* h = S.hdr + k % kPRing;
      if (state == 2) {
        if (lane == 0) {
          h->unit = -1;
          st_release_block(&S.misc[M_PUB], k + 1);
        }
        break;
      }
      const PQEntry* e = A.dq + t;
      const int unit = __ldcg(&e->unit), t0 = __ldcg(&e->t0), nt = __ldcg(&e->nt);
      // the chunk's tile descriptors (nt <= kPMaxC = 32) and the unit's q
      if (lane < nt) {
        const int4* src = reinterpret_cast<const int4*>(A.tiles + (size_t)unit * p.mpp + t0 + lane);
        int4* dst = reinterpret_cast<int4*>(S.ring_tiles + (k % kPRing) * kPMaxC + lane);
        dst[0] = __ldcg(src);
        dst[1] = __ldcg(src + 1);
      }
      {
        const int b = unit / p.Hk, kvh = unit % p.Hk;
        const uint4* qsrc = reinterpret_cast<const uint4*>(A.q + ((size_t)b * p.Hq + kvh * G) * kD);
        uint4* qdst = reinterpret_cast<uint4*>(S.ring_q + (size_t)(k % kPRing) * G * kD * 2);
        for (int i = lane; i < G * (kD / 8); i += 32) qdst[i] = __ldg(qsrc + i);
      }
      __syncwarp();
      if (lane == 0) {
        h->unit = unit;
        h->t0 = t0;
        h->nt = nt;
        h->nch = __ldcg(&e->nch);
        h->pos0 = __ldcg(&e->pos0);
        h->kin = __ldcg(&e->kin);
        st_release_block(&S.misc[M_PUB], k + 1);
      }
      __syncwarp();
    }
  } else {
    // ================================================================ consumers
    const int cw = warp - kPSel;
    uint8_t* my_slots = S.slots + (size_t)cw * nslots * kSlotB;
    uint64_t* my_full = S.full + cw * 3;
    int4* my_fifo = S.fifo + cw * kFifo;
    int n_iss = 0, n_done = 0, slot_ctr = 0, busy = 0;
    uint32_t phase = 0u;
    int src = (A.given || total_items == 0) ? 1 : 0;   // 0 score items, 1 decode chunks, 2 done
    bool failed = false;
    // score items are claimed kItemBatch at a time (one atomic on one global
    // counter per batch: per-item atomics on one address serialise); the next
    // batch is claimed when the current one is half used
    int tick = 0, tick_next = 0, tick_left = 0;
    if (src == 0 && lane == 0) {
      tick = atomicAdd(&gs[kGsScoreTicket], kItemBatch);
      tick_next = atomicAdd(&gs[kGsScoreTicket], kItemBatch);
    }
    if (src == 0) tick_left = kItemBatch;
    int ck = 0, ci = 0;   // issue position: chunk ordinal, this warp's tile within it
    int pub_seen = 0;     // chunks known to be published (read again only when the issue catches up)

    // Fill free slots (and queue park markers) ahead of the compute: score
    // items while the score ticket lasts, then this warp's tiles of the
    // published chunks.  Waits only when nothing is in flight.
    auto issue = [&]() {
      while (!failed && src != 2 && n_iss - n_done < kFifo) {
        if (src == 0) {
          if (busy == nslots) break;
          const int t = __shfl_sync(0xffffffffu, tick, 0);
          if (t >= total_items) { src = 1; continue; }
          if (--tick_left > 0) {
            ++tick;
          } else {   // the batch in hand is used up: move to the claimed one, claim another
            tick_left = kItemBatch;
            if (lane == 0) {
              tick = tick_next;
              tick_next = atomicAdd(&gs[kGsScoreTicket], kItemBatch);
            }
          }
          const int u = unit_of_item(S.items, U, t);
          const int b = u / p.Hk, kvh = u % p.Hk;
          const int L = min(__ldg(A.seq_lens + b), p.mpp * kP);
          int j0, j1;
          candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
          const int first = (t - S.items[u]) * kRows;
          const int nb = min(kRows, (j1 - j0) - first);
          const int slot = slot_ctr % nslots;
          if (lane == 0) {
            uint8_t* dst = my_slots + (size_t)slot * kSlotB;
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&my_full[slot], nb * kRowB + G * kD * 2);
            bulk_load_1d(dst, A.summ_r + (((size_t)u * p.slots) + j0 + first) * kRowE, nb * kRowB, &my_full[slot]);
            bulk_load_1d(dst + kQOff, A.q + ((size_t)b * p.Hq + kvh * G) * kD, G * kD * 2, &my_full[slot]);
            my_fifo[n_iss % kFifo] = make_int4(kScore, slot, u, first | (nb << 16));
          }
          ++n_iss; ++slot_ctr; ++busy;
        } else {
          // lane 0 reads the published count (relaxed; one acquire fence when it
          // has moved) and the warp follows it
          if (pub_seen <= ck) {
            int pub = 0;
            if (lane == 0) pub = ld_relaxed_block(&S.misc[M_PUB]);
            pub = __shfl_sync(0xffffffffu, pub, 0);
            if (pub <= ck) {
              if (n_iss > n_done) break;   // compute what is in flight first
              if (lane == 0) {
                uint32_t i = 0;
                while ((pub = ld_relaxed_block(&S.misc[M_PUB])) <= ck && ++i < kSpin) __nanosleep(32);
              }
              pub = __shfl_sync(0xffffffffu, pub, 0);
              if (pub <= ck) {
                if (lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
                failed = true;
                break;
              }
            }
            if (lane == 0) fence_acq_rel_block();
            pub_seen = pub;
            __syncwarp();   // the ring entries' contents, ordered after lane 0's acquire
          }
          const RingHdr* h = S.hdr + ck % kPRing;
          const int unit = h->unit;
          if (unit < 0) { src = 2; break; }
          const int nt = h->nt;
          const int mine = nt > cw ? (nt - cw + kPC - 1) / kPC : 0;
          if (ci < mine) {
            if (busy == nslots) break;
            const int ti = cw + kPC * ci;
            const int slot = slot_ctr % nslots;
            if (lane == 0) {
              const Tile& tl = S.ring_tiles[(ck % kPRing) * kPMaxC + ti];
              uint8_t* dst = my_slots + (size_t)slot * kSlotB;
              fence_proxy_async_smem();
              if (tl.phys >= 0) {
                const int row = (tl.phys * p.Hk + (unit % p.Hk)) * kP;
                mbar_arrive_expect_tx(&my_full[slot], 2 * kSlab);
                tma_load_3d(dst, &tmK, 0, row, 0, &my_full[slot]);
                tma_load_3d(dst + kSlab, &tmV, 0, row, 0, &my_full[slot]);
              } else {
                mbar_arrive(&my_full[slot]);
              }
              my_fifo[n_iss % kFifo] = make_int4(kTile, slot, ck, ti);
            }
            ++n_iss; ++slot_ctr; ++busy; ++ci;
          } else {
            if (lane == 0) my_fifo[n_iss % kFifo] = make_int4(kPark, -1, ck, 0);
            ++n_iss; ++ck; ci = 0;
          }
        }
      }
      __syncwarp();   // lane 0's entries are visible to the warp
    };
    // every lane observes the slot's phase (the copies' writes are then visible to it)
    auto land = [&](int slot) {
      const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&my_full[slot], (phase >> slot) & 1u, A.status));
      phase ^= 1u << slot;
      return ok;
    };

    // ---------------- phase 1: score items (no attention state is live here)
    for (;;) {
      issue();
      if (n_done == n_iss || failed) break;
      const int4 e = my_fifo[n_done % kFifo];
      if (e.x != kScore) break;   // the next entry is a tile or a park marker: phase 2
      ++n_done;
      if (!land(e.y)) {
        failed = true;
        break;
      }
      score_item<MODE>(p, A, my_slots + (size_t)e.y * kSlotB, e.z, e.w & 0xffff, e.w >> 16, lane);
      __syncwarp();   // every lane's scores (and reads of the slot) before lane 0's release of the count
      if (lane == 0) red_release_gpu_add(unit_scored + e.z, e.w >> 16);
      --busy;
    }

    // ---------------- phase 2: decode tiles and park markers
    {
      uint8_t* sp = S.pbuf + cw * 512;
      const float scale_log2 = p.scale * 1.4426950408889634f;
      const int g4 = lane >> 2, t4 = lane & 3;
      int q_unit = -1;
      uint32_t qb[8][2];
      AttnState st;
      attn_reset(st);
      while (!failed) {
        issue();
        if (n_done == n_iss) break;   // done (src == 2) or failed
        const int4 e = my_fifo[n_done % kFifo];
        ++n_done;
        if (e.x == kTile) {
          if (!land(e.y)) {
            failed = true;
            break;
          }
          const RingHdr* h = S.hdr + e.z % kPRing;
          const int unit = h->unit;
          if (unit != q_unit) {   // Q fragments (B operand: k = dim, n = head), heads >= G are zero
            q_unit = unit;
            const bool hv = g4 < G;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                S.ring_q + (size_t)(e.z % kPRing) * G * kD * 2 + (size_t)(hv ? g4 : 0) * kD * 2);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              qb[ks][0] = hv ? qrow[ks * 8 + t4] : 0u;
              qb[ks][1] = hv ? qrow[ks * 8 + 4 + t4] : 0u;
            }
          }
          const Tile tl = S.ring_tiles[(e.z % kPRing) * kPMaxC + e.w];
          if (tl.phys >= 0) attend_tile(my_slots + (size_t)e.y * kSlotB, tl, qb, scale_log2, st, sp, lane);
          __syncwarp();   // every lane is done with the slot before it is refilled
          --busy;
          continue;
        }
        if (e.x == kScore) {   // cannot follow a tile; never leave a copy unwaited
          land(e.y);
          --busy;
          continue;
        }
        // ---------------- park this warp's state of chunk k; the last warp combines
        const int k = e.z;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, off);
          st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, off);
        }
        int ok = 1;
        if (lane == 0) {   // the park buffer is free once chunk k - 1 is combined
          uint32_t i = 0;
          while (ld_relaxed_block(&S.misc[M_COMB]) < k && ++i < kSpin) __nanosleep(32);
          ok = i < kSpin;
          fence_acq_rel_block();
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
          failed = true;
          break;
        }
        __syncwarp();   // the writes below are ordered after lane 0's acquire
        float* ww = S.park + cw * G * kPartF;
        const bool w0ok = 2 * t4 < G, w1ok = 2 * t4 + 1 < G;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
          const int d = mt * 16 + g4;
          if (w0ok) {
            ww[(2 * t4) * kPartF + d] = st.o[mt][0];
            ww[(2 * t4) * kPartF + d + 8] = st.o[mt][2];
          }
          if (w1ok) {
            ww[(2 * t4 + 1) * kPartF + d] = st.o[mt][1];
            ww[(2 * t4 + 1) * kPartF + d + 8] = st.o[mt][3];
          }
        }
        if (g4 == 0) {
          if (w0ok) { ww[(2 * t4) * kPartF + kD] = st.m0; ww[(2 * t4) * kPartF + kD + 1] = st.l0; }
          if (w1ok) { ww[(2 * t4 + 1) * kPartF + kD] = st.m1; ww[(2 * t4 + 1) * kPartF + kD + 1] = st.l1; }
        }
        attn_reset(st);
        __syncwarp();
        int last = 0;
        if (lane == 0) {
          __threadfence_block();
          last = atomicAdd(&S.misc[M_PARKED], 1) == kPC - 1;
          __threadfence_block();
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();   // the other warps' parked states, ordered after lane 0's count
        if (!last) continue;
        combine_chunk(p, A, S, k, lane, unit_done);
      }
    }
    if (failed) {
      // copies still in flight must land before the CTA's shared memory goes away
      for (int i = n_done; i < n_iss; ++i) {
        const int4 f = my_fifo[i % kFifo];
        if (f.x == kScore || f.x == kTile) land(f.y);
      }
      __syncwarp();
    }
  }

  // ---- every role is done: the last CTA to leave zeroes the counters of this launch
  __syncthreads();
  if (tid == 0) {
    S.misc[M_LASTCTA] = atom_acq_rel_gpu_add(&gs[kGsExit], 1) == (int)gridDim.x - 1;
    if (S.misc[M_LASTCTA]) S.misc[M_QTAIL] = min(ld_relaxed_gpu(&gs[kGsQTail]), A.qcap);
  }
  __syncthreads();
  if (S.misc[M_LASTCTA]) {
    const int nq = S.misc[M_QTAIL];
    for (int i = tid; i < nq; i += blockDim.x) A.dq[i].flag = 0;
    for (int i = tid; i < kGsHead + kGsPerUnit * U; i += blockDim.x)
      if (i != kGsExit) gs[i] = 0;
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      gs[kGsExit] = 0;
      __threadfence();
    }
  }
}

}  // namespace

// ------------------------------------------------------------------ host

int persist_chunk_tiles(const Params&) { return kPMaxC; }

size_t persist_qcap(const Params& p) {
  const int C = persist_chunk_tiles(p);
  const size_t per_unit = std::min<size_t>(kPMaxChunksUnit, ((size_t)p.mpp + C - 1) / C);
  return (size_t)p.B * p.Hk * per_unit;
}

size_t persist_gs_bytes(const Params& p) { return ((size_t)kGsHead + kGsPerUnit * (size_t)p.B * p.Hk) * sizeof(int); }

size_t persist_partials_bytes(const Params& p) { return persist_qcap(p) * partial_stride(p.G) * sizeof(float); }

// Slots per consumer warp that fit next to the rest of the kernel's shared memory (0: none).
static int persist_slots(const Params& p) {
  for (int n = 3; n >= 2; --n)
    if (smem_plan(p.B * p.Hk, p.G, n).total <= 227 * 1024) return n;
  return 0;
}

bool persist_supported(const Params& p, bool step) {
  if (p.bypass != nullptr) return false;
  if (p.B * p.Hk > kPMaxUnits) return false;
  if ((long long)p.mpp > (long long)kPMaxC * kPMaxChunksUnit) return false;
  if (persist_slots(p) == 0) return false;
  if (step) {
    if (p.sel_mode != SA_SELECT_PER_HEAD) return false;
  }
  return true;
}

int launch_persist(const Params& p, const PArgs& A_in, const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms,
                   cudaStream_t stream) {
  PArgs A = A_in;
  A.nslots = persist_slots(p);
  if (A.nslots == 0) return SA_ERR_UNSUPPORTED;
  A.C = persist_chunk_tiles(p);
  A.qcap = (int)persist_qcap(p);
  const size_t smem = smem_plan(p.B * p.Hk, p.G, A.nslots).total;
  void (*kern)(Params, PArgs, const CUtensorMap, const CUtensorMap) =
      p.mode == SA_SUMMARY_MINMAX ? step_kernel<SA_SUMMARY_MINMAX> : step_kernel<SA_SUMMARY_MEAN>;
  if (smem_limit_at_least(reinterpret_cast<const void*>(kern), (int)smem) != cudaSuccess) return SA_ERR_CUDA;
  const cudaError_t e = launch_pdl(kern, dim3(std::max(1, num_sms)), dim3(kPThreads), smem, stream, p, A, tmK, tmV);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
