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
// Kernel 2 (decode, persistent, stream-K): the tile lists of all units are
// concatenated and every CTA takes an equal contiguous slice, so the load is
// balanced whatever the union sizes are.  A producer warp keeps a ring of
// page slots full (one lane per slot, each running on its own): it reads the
// tile descriptor (the builder already looked the page up) and issues 2-D TMA
// loads (SWIZZLE_128B, two 16 x 64 bf16 boxes per 4 KB slab of K and of V)
// that complete on the slot's "full" mbarrier.  Consumer warps take the slice's
// tiles round-robin: S = K Q^T and O^T += V^T P on mma.sync m16n8k16 (tokens x
// heads, heads padded to 8), with P split into a bf16 high part and a bf16
// residual so the product keeps ~16 mantissa bits; they release the slot on
// its "empty" mbarrier.  At the end of each unit segment the consumer warps
// merge their states; a unit split over several CTAs leaves one partial per
// CTA, and the last CTA to finish merges them in CTA order (deterministic).
#include <cuda.h>

#include <algorithm>

#include "sa_common.cuh"
#include "tiles.cuh"

namespace sa {

constexpr int kConsWarps = 4;                      // consumer warps
constexpr int kDecThreads = (kConsWarps + 1) * 32; // + one producer warp
constexpr int kMaxCtas = 1024;                     // grid cap (partial slots are sized for it)
constexpr int kMaxSlotsPerWarp = 4;                // slots <= 16
constexpr int kPart = kD + 2;                      // floats per head in a partial: O[kD], max, sum
constexpr int kSlab = kP * kD * 2;           // 4096 bytes: one page of one KV head
constexpr int kTileBytes = 2 * kSlab;        // K + V
constexpr int kBoxBytes = 16 * 64 * 2;       // one TMA box: 16 rows x 64 bf16

// ------------------------------------------------------------------ tile builder

constexpr int kBuildThreads = 1024;

__global__ void __launch_bounds__(kBuildThreads)
build_tiles_kernel(Params p, const int* __restrict__ seq_lens, const int* __restrict__ page_table,
                   const int* __restrict__ sel_idx, const int* __restrict__ sel_cnt, int gran,
                   Tile* __restrict__ tiles, int* __restrict__ ntiles, float* __restrict__ out,
                   float* __restrict__ lse, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ int flag[];  // [mpp]: page flag, then tile index
  __shared__ int scan_tmp[32];
  build_unit_tiles(p, blockIdx.y, blockIdx.x, seq_lens, page_table, sel_idx, sel_cnt, gran, tiles, ntiles, out, lse,
                   status, flag, scan_tmp);
}

// ------------------------------------------------------------------ decode

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int* page_table;
  const Tile* tiles;
  const int* ntiles;
  float* partials;   // [kMaxCtas][2][G][kPart]
  int* counters;     // [U]
  float* out;
  float* lse;
  float* logits;     // may be null
  int* status;
};

struct __align__(16) SlotInfo {
  int unit, lp, phys, pad;
  uint32_t mask[4];
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..15) of row `row` inside a K or V
  // slab written by two SWIZZLE_128B boxes of 16 rows x 128 bytes
  return (uint32_t)((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsWarps * 32) : "memory");
}

// CTA whose slice [c T / n, (c+1) T / n) holds global tile x.
__device__ __forceinline__ int cta_of(long long x, long long T, int n) {
  return (int)(((x + 1) * n + T - 1) / T) - 1;
}

__device__ __forceinline__ long long slice_lo(int c, long long T, int n) { return (long long)c * T / n; }

// Unit u with prefix[u] <= x < prefix[u + 1] (prefix non-decreasing, x < prefix[U]).
__device__ __forceinline__ int unit_of(const int* prefix, int U, long long x) {
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(Params p, DecodeArgs A, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, int nslots) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // nslots page slots (a multiple of kConsWarps), then small state
  uint8_t* s_tiles = smem;                                                   // nslots * kTileBytes
  uint8_t* s_p = s_tiles + (size_t)nslots * kTileBytes;                      // kConsWarps * 512
  float* s_w = reinterpret_cast<float*>(s_p + kConsWarps * 512);             // kConsWarps * G * kPart
  SlotInfo* s_info = reinterpret_cast<SlotInfo*>(s_w + kConsWarps * p.G * kPart);   // nslots
  uint64_t* s_full = reinterpret_cast<uint64_t*>(s_info + nslots);           // nslots
  uint64_t* s_empty = s_full + nslots;                                       // nslots
  int* s_misc = reinterpret_cast<int*>(s_empty + nslots);                    // 32 ints
  int* s_prefix = s_misc + 32;                                               // U + 1

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G;
  const int U = p.B * p.Hk;

  if (tid == 0) {
    for (int i = 0; i < nslots; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 1);
    }
    fence_mbar_init();
    s_misc[16] = 0;
  }
  // prefix over the units' tile counts (block-wide scan)
  {
    const int per = (U + blockDim.x - 1) / blockDim.x;
    const int a = min(U, tid * per), e = min(U, a + per);
    int cnt = 0;
    for (int i = a; i < e; ++i) cnt += A.ntiles[i];
    int x = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_misc[warp] = x;
    __syncthreads();
    int before = x - cnt;
    for (int w2 = 0; w2 < warp; ++w2) before += s_misc[w2];
    for (int i = a; i < e; ++i) {
      s_prefix[i] = before;
      before += A.ntiles[i];
    }
    if (tid == blockDim.x - 1) s_prefix[U] = before;
  }
  __syncthreads();
  const long long T = s_prefix[U];
  // slice over n_eff = min(grid, T) CTAs so that every slice is non-empty: the
  // split-unit merge counts one arrival per CTA index between two slices
  const int nC = (int)min((long long)gridDim.x, T), c = blockIdx.x;
  if (c >= nC) return;
  const long long lo = slice_lo(c, T, nC), hi = slice_lo(c + 1, T, nC);
  if (lo >= hi) return;
  const int n_local = (int)(hi - lo);

  // ------------------------------------------------------------ producer warp
  // Lane j (< nslots) owns slot j and issues that slot's uses in order.  The
  // slice's tiles are handed out in order to whichever slots are free, so a
  // tile that lands late holds back only its own slot.  Descriptors come in
  // batches of 32 (one per lane, the next batch loaded ahead) and are passed
  // to the issuing lane by shuffle.
  if (warp == kConsWarps) {
    const bool owner = lane < nslots;
    int use = 0, next = 0, dbase = 0;
    int4 dA0, dB0;
    uint4 dA1, dB1;
    auto load_desc = [&](int base_, int4& w0, uint4& w1) {
      const int i = base_ + lane;
      if (i < n_local) {
        const long long t = lo + i;
        const int uu = unit_of(s_prefix, U, t);
        const Tile* tp = A.tiles + (size_t)uu * p.mpp + (t - s_prefix[uu]);
        w0 = __ldg(reinterpret_cast<const int4*>(tp));
        w1 = __ldg(reinterpret_cast<const uint4*>(&tp->mask[0]));
        w0.z = uu;   // the unit rides in a pad field
      } else {
        w0 = make_int4(0, -1, 0, 0);
        w1 = make_uint4(0, 0, 0, 0);
      }
    };
    load_desc(0, dA0, dA1);
    load_desc(32, dB0, dB1);
    uint32_t spins = 0;
    while (next < n_local) {
      const bool free_slot = owner && (use == 0 || mbar_test_wait(&s_empty[lane], (use - 1) & 1));
      const unsigned fm = __ballot_sync(0xffffffffu, free_slot);
      const int n_issue = min(__popc(fm), min(32 - (next - dbase), n_local - next));
      const int rank = __popc(fm & ((1u << lane) - 1u));
      const bool mine = free_slot && rank < n_issue;
      const int src = next - dbase + (mine ? rank : 0);
      int4 w0;
      uint4 w1;
      w0.x = __shfl_sync(0xffffffffu, dA0.x, src);
      w0.y = __shfl_sync(0xffffffffu, dA0.y, src);
      w0.z = __shfl_sync(0xffffffffu, dA0.z, src);
      w1.x = __shfl_sync(0xffffffffu, dA1.x, src);
      w1.y = __shfl_sync(0xffffffffu, dA1.y, src);
      w1.z = __shfl_sync(0xffffffffu, dA1.z, src);
      w1.w = __shfl_sync(0xffffffffu, dA1.w, src);
      if (mine) {
        const int slot = lane, u = w0.z;
        const int phys = (w0.y >= 0 && w0.y < p.num_pages) ? w0.y : -1;
        SlotInfo info;
        info.unit = u;
        info.lp = w0.x;
        info.phys = phys;
        info.pad = 0;
        info.mask[0] = w1.x; info.mask[1] = w1.y; info.mask[2] = w1.z; info.mask[3] = w1.w;
        s_info[slot] = info;
        if (phys >= 0) {
          uint8_t* dst = s_tiles + (size_t)slot * kTileBytes;
          const int row = (phys * p.Hk + (u % p.Hk)) * kP;
          mbar_arrive_expect_tx(&s_full[slot], kTileBytes);
          tma_load_2d(dst, &tmK, 0, row, &s_full[slot]);
          tma_load_2d(dst + kBoxBytes, &tmK, 64, row, &s_full[slot]);
          tma_load_2d(dst + kSlab, &tmV, 0, row, &s_full[slot]);
          tma_load_2d(dst + kSlab + kBoxBytes, &tmV, 64, row, &s_full[slot]);
        } else {
          mbar_arrive(&s_full[slot]);
        }
        ++use;
      }
      next += n_issue;
      if (next - dbase >= 32) {   // move to the next batch and load the one after it
        dA0 = dB0;
        dA1 = dB1;
        dbase += 32;
        load_desc(dbase + 32, dB0, dB1);
      }
      if (n_issue == 0 && ++spins > (1u << 28)) {   // bounded: consumers stopped releasing slots
        set_status(A.status, SA_ERR_TIMEOUT);
        break;
      }
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const float scale_log2 = p.scale * 1.4426950408889634f;
  const int g4 = lane >> 2, t4 = lane & 3;
  uint8_t* sp = s_p + warp * 512;
  const uint32_t sp_hi = smem_u32(sp), sp_lo = sp_hi + 256;
  const int tc = tid;   // consumer thread index == head-dim index in the merges (kConsWarps * 32 == kD)
  int uses[kMaxSlotsPerWarp];   // completed uses of each of this warp's slots
#pragma unroll
  for (int m = 0; m < kMaxSlotsPerWarp; ++m) uses[m] = 0;

  for (int u = unit_of(s_prefix, U, lo); u < U && s_prefix[u] < hi; ++u) {
    const long long ub = s_prefix[u], ue = s_prefix[u + 1];
    const long long sb = max(lo, ub), se = min(hi, ue);
    if (sb >= se) continue;
    const int b = u / p.Hk, kvh = u % p.Hk;

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
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[8][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

    const int seg_size = (int)(se - sb);
    // poll this warp's slots (warp, warp + kConsWarps, ...) and take whichever
    // has landed; a slot holding a later unit's tile is left for its segment
    bool held[kMaxSlotsPerWarp];
#pragma unroll
    for (int m = 0; m < kMaxSlotsPerWarp; ++m) held[m] = false;
    uint32_t spins = 0;
    while (true) {
#pragma unroll
      for (int m = 0; m < kMaxSlotsPerWarp; ++m) {
        const int slot = warp + kConsWarps * m;
        if (slot >= nslots || held[m]) continue;
        const bool ready = __shfl_sync(0xffffffffu, (int)mbar_test_wait(&s_full[slot], uses[m] & 1), 0) != 0;
        if (!ready) continue;
        const SlotInfo* info = s_info + slot;
        if (info->unit != u) {
          held[m] = true;
          continue;
        }
        if (info->phys >= 0) {
          const uint32_t sK = smem_u32(s_tiles + (size_t)slot * kTileBytes);
          const uint32_t sV = sK + kSlab;
          // S = K Q^T  (rows = tokens, cols = heads), two accumulators to halve the chain
          float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb2[4] = {0.f, 0.f, 0.f, 0.f};
          {
            const int mi = lane >> 3, r = lane & 7;
            const int row = (mi & 1) * 8 + r;
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
              uint32_t a0, a1, a2, a3;
              ldsm_x4(sK + swz(row, ks * 2 + (mi >> 1)), a0, a1, a2, a3);
              mma_bf16_16816(sa, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
              ldsm_x4(sK + swz(row, (ks + 1) * 2 + (mi >> 1)), a0, a1, a2, a3);
              mma_bf16_16816(sb2, a0, a1, a2, a3, qb[ks + 1][0], qb[ks + 1][1]);
            }
          }
          const float s0 = sa[0] + sb2[0], s1 = sa[1] + sb2[1], s2 = sa[2] + sb2[2], s3 = sa[3] + sb2[3];
          // masks: tokens g4 and g4 + 8, heads 2 t4 and 2 t4 + 1
          const uint32_t mb0 = (info->mask[g4 >> 2] >> (8 * (g4 & 3))) & 0xffu;
          const uint32_t mb1 = (info->mask[2 + (g4 >> 2)] >> (8 * (g4 & 3))) & 0xffu;
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
            const int base_tok = info->lp * kP;
            const size_t hs = (size_t)p.mpp * kP;
            const size_t row0 = ((size_t)b * p.Hq + kvh * G) * hs;
            if (v00) A.logits[row0 + h0 * hs + base_tok + g4] = s0 * p.scale;
            if (v01) A.logits[row0 + h1 * hs + base_tok + g4] = s1 * p.scale;
            if (v10) A.logits[row0 + h0 * hs + base_tok + g4 + 8] = s2 * p.scale;
            if (v11) A.logits[row0 + h1 * hs + base_tok + g4 + 8] = s3 * p.scale;
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
        }
        __syncwarp();   // all lanes done reading the slot (and the P buffer)
        if (lane == 0) {
          mbar_arrive(&s_empty[slot]);
          atomicAdd(&s_misc[16], 1);
        }
        ++uses[m];
      }
      const int done = __shfl_sync(0xffffffffu, *reinterpret_cast<volatile int*>(&s_misc[16]), 0);
      if (done >= seg_size) break;
      if (++spins > (1u << 26)) {   // bounded: a copy never landed
        if (lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
        break;
      }
    }
    // row sums over the 8 lanes that share t4
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // ---- merge the consumer warps' states: s_w[warp][head][kPart]
    {
      float* ww = s_w + warp * G * kPart;
      const bool w0ok = 2 * t4 < G, w1ok = 2 * t4 + 1 < G;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int d = mt * 16 + g4;
        if (w0ok) {
          ww[(2 * t4) * kPart + d] = o[mt][0];
          ww[(2 * t4) * kPart + d + 8] = o[mt][2];
        }
        if (w1ok) {
          ww[(2 * t4 + 1) * kPart + d] = o[mt][1];
          ww[(2 * t4 + 1) * kPart + d + 8] = o[mt][3];
        }
      }
      if (g4 == 0) {
        if (w0ok) { ww[(2 * t4) * kPart + kD] = m0; ww[(2 * t4) * kPart + kD + 1] = l0; }
        if (w1ok) { ww[(2 * t4 + 1) * kPart + kD] = m1; ww[(2 * t4 + 1) * kPart + kD + 1] = l1; }
      }
    }
    consumer_sync();
    const bool whole = ub >= lo && ue <= hi;
    const int pslot = ub <= lo ? 0 : 1;   // this CTA's first segment, or its last
    float* part = A.partials + ((size_t)c * 2 + pslot) * G * kPart;
    for (int g = 0; g < G; ++g) {
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kConsWarps; ++ww) M = fmaxf(M, s_w[(ww * G + g) * kPart + kD]);
      float acc = 0.f, l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int ww = 0; ww < kConsWarps; ++ww) {
          const float mw = s_w[(ww * G + g) * kPart + kD];
          const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
          acc += f * s_w[(ww * G + g) * kPart + tc];
          l += f * s_w[(ww * G + g) * kPart + kD + 1];
        }
      }
      if (whole) {
        const size_t row = (size_t)b * p.Hq + kvh * G + g;
        A.out[row * kD + tc] = l > 0.f ? acc / l : 0.f;
        if (tc == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
      } else {
        part[g * kPart + tc] = acc;
        if (tc == 0) {
          part[g * kPart + kD] = M;
          part[g * kPart + kD + 1] = l;
        }
      }
    }
    if (!whole) {
      __threadfence();
      consumer_sync();
      const int c_first = cta_of(ub, T, nC), c_last = cta_of(ue - 1, T, nC);
      if (tc == 0) {
        const int prev = atomicAdd(&A.counters[u], 1);
        s_misc[0] = (prev == c_last - c_first);
      }
      consumer_sync();
      if (s_misc[0]) {
        __threadfence();
        // Merge the CTAs' partials in CTA order.  The (max, sum) of every
        // (partial, head) is staged in shared memory (s_w is free here) so
        // the loads overlap instead of forming a dependent chain.
        const int np = c_last - c_first + 1;
        const int chunk = 256 / G;            // partials per staging round (2 x 256 floats fit s_w)
        float* sm_a = s_w;                    // [chunk][G]: max, then weight
        float* sm_b = s_w + 256;              // [chunk][G]: sum
        float* sm_M = reinterpret_cast<float*>(s_misc + 8);   // [G]: running max
        if (tc < G) sm_M[tc] = -INFINITY;
        consumer_sync();
        for (int base = 0; base < np; base += chunk) {
          const int nb = min(np - base, chunk);
          for (int idx = tc; idx < nb * G; idx += kConsWarps * 32) {
            const int cc = c_first + base + idx / G, g = idx % G;
            const int ps = ub <= slice_lo(cc, T, nC) ? 0 : 1;
            sm_a[idx] = __ldcg(A.partials + (((size_t)cc * 2 + ps) * G + g) * kPart + kD);
          }
          consumer_sync();
          if (tc < G) {
            float M = sm_M[tc];
            for (int j = 0; j < nb; ++j) M = fmaxf(M, sm_a[j * G + tc]);
            sm_M[tc] = M;
          }
          consumer_sync();
        }
        float accs[kMaxG], ls[kMaxG];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) { accs[g] = 0.f; ls[g] = 0.f; }
        for (int base = 0; base < np; base += chunk) {
          const int nb = min(np - base, chunk);
          for (int idx = tc; idx < nb * G; idx += kConsWarps * 32) {
            const int cc = c_first + base + idx / G, g = idx % G;
            const int ps = ub <= slice_lo(cc, T, nC) ? 0 : 1;
            const float* pc = A.partials + (((size_t)cc * 2 + ps) * G + g) * kPart;
            const float mc = __ldcg(pc + kD), M = sm_M[g];
            sm_a[idx] = (mc == -INFINITY || M == -INFINITY) ? 0.f : exp2f(mc - M);
            sm_b[idx] = __ldcg(pc + kD + 1);
          }
          consumer_sync();
#pragma unroll 4
          for (int j = 0; j < nb; ++j) {
            const int cc = c_first + base + j;
            const int ps = ub <= slice_lo(cc, T, nC) ? 0 : 1;
            const float* pc = A.partials + ((size_t)cc * 2 + ps) * G * kPart;
#pragma unroll
            for (int g = 0; g < kMaxG; ++g) {
              if (g < G) {
                const float f = sm_a[j * G + g];
                accs[g] += f * __ldcg(pc + g * kPart + tc);
                ls[g] += f * sm_b[j * G + g];
              }
            }
          }
          consumer_sync();
        }
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) {
          if (g < G) {
            const size_t row = (size_t)b * p.Hq + kvh * G + g;
            A.out[row * kD + tc] = ls[g] > 0.f ? accs[g] / ls[g] : 0.f;
            if (tc == 0) A.lse[row] = ls[g] > 0.f ? (sm_M[g] + log2f(ls[g])) * 0.6931471805599453f : -INFINITY;
          }
        }
        if (tc == 0) A.counters[u] = 0;
      }
    }
    if (tc == 0) s_misc[16] = 0;   // tiles-done counter of the next segment
    consumer_sync();   // s_w and s_misc are reused by the next segment
  }
}

size_t decode_smem_bytes_n(int U, int G, int nslots) {
  return 1024 + (size_t)nslots * kTileBytes + kConsWarps * 512 + (size_t)kConsWarps * G * kPart * 4 +
         nslots * sizeof(SlotInfo) + 2 * nslots * 8 + 32 * 4 + (size_t)(U + 1) * 4;
}

// Slot count: the largest multiple of kConsWarps (<= 16) that still lets two
// CTAs share an SM; at least kConsWarps.
int decode_slots(int U, int G) {
  const size_t per_sm = 228 * 1024, reserve = 1024;
  int best = kConsWarps;
  for (int n = kConsWarps; n <= 16; n += kConsWarps)
    if (2 * (decode_smem_bytes_n(U, G, n) + reserve) <= per_sm) best = n;
  return best;
}

size_t decode_smem_bytes(int U) { return decode_smem_bytes_n(U, kMaxG, kConsWarps); }

size_t decode_partials_bytes(const Params& p) { return (size_t)kMaxCtas * 2 * p.G * kPart * sizeof(float); }

size_t tiles_bytes(const Params& p) { return (size_t)p.B * p.Hk * p.mpp * sizeof(Tile); }

int launch_build_tiles(const Params& p, const int* seq_lens, const int* page_table, const int* sel_idx,
                       const int* sel_cnt, int gran, void* tiles, int* ntiles, float* out, float* lse, int* status,
                       cudaStream_t stream) {
  const size_t smem = (size_t)p.mpp * sizeof(int);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(build_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(p.Hk, p.B);
  const cudaError_t e = launch_pdl(build_tiles_kernel, grid, dim3(kBuildThreads), smem, stream, p, seq_lens,
                                   page_table, sel_idx, sel_cnt, gran, static_cast<Tile*>(tiles), ntiles, out, lse,
                                   status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int launch_decode(const Params& p, const void* q, const int* page_table, const void* tiles, const int* ntiles,
                  float* partials, int* counters, float* out, float* lse, float* logits, int* status,
                  const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  const int U = p.B * p.Hk;
  const int nslots = decode_slots(U, p.G);
  const size_t smem = decode_smem_bytes_n(U, p.G, nslots);
  if (smem > 227 * 1024) return SA_ERR_UNSUPPORTED;
  cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel, kDecThreads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int grid = std::min(kMaxCtas, num_sms * per_sm);
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
  const cudaError_t e = launch_pdl(decode_kernel, dim3(grid), dim3(kDecThreads), smem, stream, p, A, tmK, tmV, nslots);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
