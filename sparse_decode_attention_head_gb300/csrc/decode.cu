// Steps a4 + a5 + a6: paged-gather split-K decode attention over the dense set
// I (sinks + recent window) and each head's selected set J_h, merged exactly
// with the log-sum-exp identity.
//
// HGCA (review, "What carries the argument") attends a recent window densely
// and selected older entries sparsely and fuses the two partial outputs with
//   O = (e^lse_I O_I + e^lse_J O_J) / (e^lse_I + e^lse_J).
// The identity holds for any partition, so here the attended rows of one KV
// head are cut into chunks of whole pages, each chunk leaves a partial
// (max, sum, unnormalised O) per query head, and the chunks of a unit are
// merged with the same identity, in chunk order, stabilised by the running
// maximum (the review's comment on Sec. 3.3).
//
// Kernel 1 (tile builder, one CTA per (sequence, KV head, window of 4096
// pages)): the union over the G query heads of the pages to read, as an
// ascending list of tiles per window; a tile is one 16-token page with a
// G-bit head mask per token, so the rows a GQA group shares are read once
// (SPIN abstract / Fig. 6: paged KV substrate).
//
// Kernel 2 (decode, persistent, dynamically scheduled): the tile lists are cut
// into chunks of C tiles that never cross a unit; CTA c starts on chunk c and
// takes further chunks from a global ticket counter, so CTAs whose pages land
// faster take more chunks.  A producer warp keeps a ring of page slots full
// (one lane per slot): it reads the tile descriptor (the builder already
// looked the page up) and issues 2-D TMA loads (SWIZZLE_128B, two 16 x 64
// bf16 boxes per 4 KB slab of K and of V) that complete on the slot's "full"
// mbarrier.  Consumer warps take the landed slots of their current chunk:
// S = K Q^T and O^T += V^T P on mma.sync m16n8k16 (tokens x heads, heads
// padded to 8), with P split into a bf16 high part and a bf16 residual so the
// product keeps ~16 mantissa bits; they release the slot on its "empty"
// mbarrier.  A warp that has done its share of a chunk parks its state and
// moves on; the last warp to park combines the four states into the chunk
// partial.
//
// Kernel 3 (merge, one CTA per (query head, unit)): the chain merge of the
// unit's chunk partials.  Units held in one chunk are finished by kernel 2.
#include <cuda.h>

#include <algorithm>

#include "sa_common.cuh"
#include "tiles.cuh"

namespace sa {

constexpr int kConsWarps = 4;                      // consumer warps
constexpr int kDecThreads = (kConsWarps + 1) * 32; // + one producer warp
constexpr int kMaxCtas = 512;                      // grid cap (partial slots are sized for it)
constexpr int kChunksPerCta = 3;                   // chunk size: about this many chunks per CTA ...
constexpr int kMinChunk = 8;                       // ... but at least this many tiles
constexpr int kChunkRing = 32;                     // published chunks not yet finished (> slots)
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
                   Tile* __restrict__ tiles, int* __restrict__ ntiles, int* status, int* ticket) {
  pdl_wait();
  pdl_trigger();
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) *ticket = 0;   // the decode's chunk tickets
  extern __shared__ int smem_b[];   // build_smem_bytes(mpp): window flags, then window masks
  __shared__ int scan_tmp[32];
  const int win = min(p.mpp, kWinPages);
  const int kvh = blockIdx.x, b = blockIdx.y;
  const size_t h0 = (size_t)b * p.Hq + kvh * p.G;
  const uint32_t active = unit_active_heads(p, b, kvh);
  build_unit_tiles<kBuildThreads>(p, b, kvh, seq_lens, page_table, sel_idx + h0 * p.kcap, sel_cnt + h0, gran, tiles,
                                  ntiles, status, smem_b, reinterpret_cast<uint32_t*>(smem_b + win),
                                  scan_tmp, active, blockIdx.z, 1);
}

// ------------------------------------------------------------------ decode

struct DecodeArgs {
  const __nv_bfloat16* q;
  const int* page_table;
  const Tile* tiles;
  const int* ntiles;
  float* partials;   // [chunks][partial_stride(G)]: per chunk O[G][kD], max[G], sum[G]
  int nwin;          // tile-list segments (windows) per unit
  int* ticket;       // chunk ticket counter (zeroed by the tile builder)
  float* out;
  float* lse;
  float* logits;     // may be null
  int* status;
};

struct __align__(16) SlotInfo {
  int unit, lp, phys, seq;   // seq: the CTA's chunk ordinal the tile belongs to
  uint32_t mask[4];
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  // byte offset of 16-byte chunk `chunk` (0..15) of row `row` inside a K or V
  // slab written by two SWIZZLE_128B boxes of 16 rows x 128 bytes
  return (uint32_t)((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}


// Chunk c of the unit-major chunk list: unit, position in the unit, tiles.
struct ChunkInfo {
  int unit;   // -1: no more chunks
  int kin;    // chunk index within the unit
  int nch;    // chunks of the unit
  int t0;     // first tile (within the unit's list)
  int nt;     // tiles in the chunk
  int pad[3];
};

// Unit u with prefix[u] <= x < prefix[u + 1] (prefix non-decreasing, x < prefix[U]).
__device__ __forceinline__ int unit_of(const int* prefix, int U, long long x) {
  int lo = 0, hi = U;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}


__device__ __forceinline__ int ld_volatile(const int* x) { return *reinterpret_cast<const volatile int*>(x); }
// CTA-scope acquire load / release store (ordering the chunk ring between
// the producer warp and the consumer warps)
__device__ __forceinline__ int ld_acquire_cta(const int* x) {
  int v;
  asm volatile("ld.acquire.cta.b32 %0, [%1];" : "=r"(v) : "l"(x) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta(int* x, int v) {
  asm volatile("st.release.cta.b32 [%0], %1;" ::"l"(x), "r"(v) : "memory");
}

// LOGITS: the instantiation that also writes every attended logit (A.logits,
// for the score tables); the plain decode carries none of that code.
template <bool LOGITS>
__global__ void __launch_bounds__(kDecThreads, 2)
decode_kernel(Params p, DecodeArgs A, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, int nslots) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int G = p.G;
  const int U = p.B * p.Hk;
  const int NW = A.nwin;
  const int SG = U * NW;   // tile-list segments: unit u, window w is segment u * NW + w
  // nslots page slots (a multiple of kConsWarps), then small state
  uint8_t* s_tiles = smem;                                                   // nslots * kTileBytes
  uint8_t* s_p = s_tiles + (size_t)nslots * kTileBytes;                      // kConsWarps * 512
  float* s_w = reinterpret_cast<float*>(s_p + kConsWarps * 512);             // kConsWarps * G * kPart
  SlotInfo* s_info = reinterpret_cast<SlotInfo*>(s_w + kConsWarps * G * kPart);   // nslots
  ChunkInfo* s_chunk = reinterpret_cast<ChunkInfo*>(s_info + nslots);       // kChunkRing
  int* s_assign = reinterpret_cast<int*>(s_chunk + kChunkRing);             // kChunkRing * kConsWarps
  uint64_t* s_full = reinterpret_cast<uint64_t*>(s_assign + kChunkRing * kConsWarps);   // nslots
  uint64_t* s_empty = s_full + nslots;                                       // nslots
  int* s_misc = reinterpret_cast<int*>(s_empty + nslots);                    // 32 ints
  int* s_prefix = s_misc + 32;                                               // SG + 1: tiles before segment s
  int* s_cprefix = s_prefix + SG + 1;                                        // SG + 1: chunks before segment s
  uint8_t* s_umask = reinterpret_cast<uint8_t*>(s_cprefix + SG + 1);        // U bytes: heads left out (bypass)
  // s_misc: [17] chunks published, [18] chunks combined, [19] chunks fully
  // issued, [20] consumer warps parked on the current chunk

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    for (int i = 0; i < nslots; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 1);
    }
    fence_mbar_init();
    s_misc[17] = 0;
    s_misc[18] = 0;
    s_misc[19] = 0;
    s_misc[20] = 0;
  }
  // heads answered by the sparsity bypass: their rows are not written.  The
  // flags are complete before this kernel starts (a call input, or written
  // by the step's score kernel, which the tile builder waited for), so they
  // are read before the wait for the tile builder.
  if (p.bypass != nullptr)
    for (int i = tid; i < U; i += blockDim.x) {
      int m = 0;
      for (int g = 0; g < G; ++g) m |= (p.bypass[(size_t)i * G + g] != 0 ? 1 : 0) << g;
      s_umask[i] = (uint8_t)m;
    }
  pdl_wait();
  pdl_trigger();
  // prefix over the segments' tile counts (block-wide scan); the chunk size
  // follows from the total so that every CTA derives the same chunk list
  const int per = (SG + blockDim.x - 1) / blockDim.x;
  const int a = min(SG, tid * per), e = min(SG, a + per);
  {
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
    if (tid == blockDim.x - 1) s_prefix[SG] = before;
  }
  __syncthreads();
  const int T = s_prefix[SG];
  const int C = max(kMinChunk, (T + kChunksPerCta * (int)gridDim.x - 1) / (kChunksPerCta * (int)gridDim.x));
  {
    int cnt = 0;
    for (int i = a; i < e; ++i) cnt += (s_prefix[i + 1] - s_prefix[i] + C - 1) / C;
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
      s_cprefix[i] = before;
      before += (s_prefix[i + 1] - s_prefix[i] + C - 1) / C;
    }
    if (tid == blockDim.x - 1) s_cprefix[SG] = before;
  }
  __syncthreads();
  const int NCH = s_cprefix[SG];
  const int PS = partial_stride(G);

  // ------------------------------------------------------------ producer warp
  // Takes chunks from the global ticket counter (one taken ahead) and
  // publishes each in the chunk ring before issuing its tiles.  Lane j
  // (< nslots) owns slot j and issues that slot's uses in order; a chunk's
  // tiles go to whichever slots are free, so a tile that lands late holds
  // back only its own slot.  Descriptors (one per lane, up to 32 at a time)
  // reach the issuing lane by shuffle.  Once a chunk is fully issued, the
  // number of its tiles each consumer warp received (slot j belongs to warp
  // j mod kConsWarps) is published, so every warp knows when its share is done.
  if (warp == kConsWarps) {
    const bool owner = lane < nslots;
    int use = 0;
    // K / V pages are read once: they should not push the partials, tile
    // lists and summaries out of L2
    const uint64_t kv_policy = l2_evict_first();
    auto chunk_info = [&](int t) {
      ChunkInfo c;
      c.unit = -1;
      c.kin = c.nch = c.t0 = c.nt = 0;
      c.pad[0] = c.pad[1] = c.pad[2] = 0;
      if (t < NCH) {
        const int sg = unit_of(s_cprefix, SG, t);   // segment holding chunk t
        const int u = sg / NW;
        const int kseg = t - s_cprefix[sg];          // chunk within the segment
        c.unit = u;
        c.kin = t - s_cprefix[u * NW];
        c.nch = s_cprefix[(u + 1) * NW] - s_cprefix[u * NW];
        c.t0 = (sg - u * NW) * kWinPages + kseg * C;   // entry within the unit's tile array
        c.nt = min(C, s_prefix[sg + 1] - s_prefix[sg] - kseg * C);
      }
      return c;
    };
    // descriptors of tiles [b0, b0 + 32) of chunk c, one per lane
    auto load_desc = [&](const ChunkInfo& c, int b0, int4& w0, uint4& w1) {
      w0 = make_int4(0, -1, 0, 0);
      w1 = make_uint4(0, 0, 0, 0);
      if (c.unit >= 0 && b0 + lane < c.nt) {
        const Tile* t = A.tiles + (size_t)c.unit * p.mpp + c.t0 + b0 + lane;
        w0 = __ldg(reinterpret_cast<const int4*>(t));
        w1 = __ldg(reinterpret_cast<const uint4*>(&t->mask[0]));
      }
    };
    // CTA c starts on chunk c; later chunks come from the ticket counter
    ChunkInfo ci = chunk_info(blockIdx.x);
    int4 dA0;
    uint4 dA1;
    load_desc(ci, 0, dA0, dA1);
    uint32_t spins = 0;
    bool stop = false;
    for (int k = 0; !stop; ++k) {
      // ring space: the consumers have finished chunk k - kChunkRing
      while (k >= kChunkRing && ld_acquire_cta(&s_misc[18]) <= k - kChunkRing) {
        if (++spins > (1u << 28)) {
          if (lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
          ci.unit = -1;
          break;
        }
      }
      if (lane == 0) {
        s_chunk[k % kChunkRing] = ci;
        st_release_cta(&s_misc[17], k + 1);
      }
      __syncwarp();
      if (ci.unit < 0) break;
      // the next chunk's ticket is taken now and read (its descriptors
      // fetched) the first time this chunk waits for a free slot
      int nxt = 0;
      if (lane == 0) nxt = (int)gridDim.x + atomicAdd(A.ticket, 1);
      bool have_next = false;
      int asg[kConsWarps];
#pragma unroll
      for (int w = 0; w < kConsWarps; ++w) asg[w] = 0;
      ChunkInfo cn;
      int4 dB0;
      uint4 dB1;
      auto fetch_next = [&]() {
        cn = chunk_info(__shfl_sync(0xffffffffu, nxt, 0));
        load_desc(cn, 0, dB0, dB1);
        have_next = true;
      };
      for (int b0 = 0; b0 < ci.nt && !stop; b0 += 32) {
        const int nb = min(32, ci.nt - b0);
        int4 dw0 = dA0;
        uint4 dw1 = dA1;
        if (b0 > 0) load_desc(ci, b0, dw0, dw1);
        int next = 0;
        while (next < nb) {
          const bool free_slot = owner && (use == 0 || mbar_test_wait(&s_empty[lane], (use - 1) & 1));
          const unsigned fm = __ballot_sync(0xffffffffu, free_slot);
          const int n_issue = min(__popc(fm), nb - next);
          const int rank = __popc(fm & ((1u << lane) - 1u));
          const bool mine = free_slot && rank < n_issue;
          const int src = next + (mine ? rank : 0);
          const int lp = __shfl_sync(0xffffffffu, dw0.x, src);
          const int ph = __shfl_sync(0xffffffffu, dw0.y, src);
          uint4 w1;
          w1.x = __shfl_sync(0xffffffffu, dw1.x, src);
          w1.y = __shfl_sync(0xffffffffu, dw1.y, src);
          w1.z = __shfl_sync(0xffffffffu, dw1.z, src);
          w1.w = __shfl_sync(0xffffffffu, dw1.w, src);
          if (mine) {
            const int slot = lane;
            const int phys = (ph >= 0 && ph < p.num_pages) ? ph : -1;
            SlotInfo info;
            info.unit = ci.unit;
            info.lp = lp;
            info.phys = phys;
            info.seq = k;
            info.mask[0] = w1.x; info.mask[1] = w1.y; info.mask[2] = w1.z; info.mask[3] = w1.w;
            s_info[slot] = info;
            if (phys >= 0) {
              uint8_t* dst = s_tiles + (size_t)slot * kTileBytes;
              const int row = (phys * p.Hk + (ci.unit % p.Hk)) * kP;
              mbar_arrive_expect_tx(&s_full[slot], kTileBytes);
              tma_load_3d_hint(dst, &tmK, 0, row, 0, &s_full[slot], kv_policy);
              tma_load_3d_hint(dst + kSlab, &tmV, 0, row, 0, &s_full[slot], kv_policy);
            } else {
              mbar_arrive(&s_full[slot]);
            }
            ++use;
          }
          next += n_issue;
          {
            const unsigned im = __ballot_sync(0xffffffffu, mine);
#pragma unroll
            for (int w = 0; w < kConsWarps; ++w) asg[w] += __popc(im & (0x11111111u << w));
          }
          if (n_issue == 0) {
            if (!have_next) fetch_next();
            if (++spins > (1u << 28)) {   // bounded: consumers stopped releasing slots
              if (lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
              stop = true;
              break;
            }
          }
        }
      }
      if (stop) {   // tell the consumers there is nothing more
        if (lane == 0) {
          ChunkInfo end;
          end.unit = -1;
          s_chunk[(k + 1) % kChunkRing] = end;
          st_release_cta(&s_misc[17], k + 2);
        }
        break;
      }
      if (lane == 0) {
#pragma unroll
        for (int w = 0; w < kConsWarps; ++w) s_assign[(k % kChunkRing) * kConsWarps + w] = asg[w];
        st_release_cta(&s_misc[19], k + 1);
      }
      if (!have_next) fetch_next();
      ci = cn;
      dA0 = dB0;
      dA1 = dB1;
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  // Each warp runs through the chunks on its own: it takes the landed slots
  // of the current chunk, and once it has processed its share it parks its
  // state (O, max, sum per head) in s_w and moves on.  The last warp to park
  // a chunk combines the parked states and writes the chunk's partial (or the
  // output, for a unit held in one chunk); parking the next chunk waits for
  // that combine, so the warps are never more than one chunk apart.
  const float scale_log2 = p.scale * 1.4426950408889634f;
  const int g4 = lane >> 2, t4 = lane & 3;
  uint8_t* sp = s_p + warp * 512;
  const uint32_t sp_hi = smem_u32(sp), sp_lo = sp_hi + 256;
  int uses[kMaxSlotsPerWarp];   // completed uses of each of this warp's slots
#pragma unroll
  for (int m = 0; m < kMaxSlotsPerWarp; ++m) uses[m] = 0;
  int q_unit = -1;
  uint32_t qb[8][2];

  // bounded wait (lane 0 polls, the warp follows) until *x > v; false on timeout
  auto wait_gt = [&](const int* x, int v) {
    int ok = 1;
    if (lane == 0) {
      uint32_t spins = 0;
      while (ld_acquire_cta(x) <= v) {
        if (++spins > (1u << 26)) { ok = 0; break; }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    if (!ok && lane == 0) set_status(A.status, SA_ERR_TIMEOUT);
    return ok != 0;
  };

  for (int k = 0;; ++k) {
    if (!wait_gt(&s_misc[17], k)) break;   // chunk k published
    const ChunkInfo ci = s_chunk[k % kChunkRing];
    if (ci.unit < 0) break;
    const int u = ci.unit;
    const int b = u / p.Hk, kvh = u % p.Hk;

    if (u != q_unit) {   // Q fragments (B operand: k = dim, n = head), heads >= G are zero
      q_unit = u;
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

    // poll this warp's slots (warp, warp + kConsWarps, ...) and take whichever
    // has landed; a slot holding a later chunk's tile is left for that chunk
    bool held[kMaxSlotsPerWarp];
#pragma unroll
    for (int m = 0; m < kMaxSlotsPerWarp; ++m) held[m] = false;
    int done = 0;
    uint32_t spins = 0;
    while (true) {
#pragma unroll
      for (int m = 0; m < kMaxSlotsPerWarp; ++m) {
        const int slot = warp + kConsWarps * m;
        if (slot >= nslots || held[m]) continue;
        const bool ready = __shfl_sync(0xffffffffu, (int)mbar_test_wait(&s_full[slot], uses[m] & 1), 0) != 0;
        if (!ready) continue;
        const SlotInfo* info = s_info + slot;
        if (info->seq != k) {
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
          if (LOGITS) {
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
        if (lane == 0) mbar_arrive(&s_empty[slot]);
        ++uses[m];
        ++done;
      }
      // this warp's share of the chunk is known once the chunk is fully issued
      int fin = 0;
      if (lane == 0 && ld_acquire_cta(&s_misc[19]) > k)
        fin = done >= s_assign[(k % kChunkRing) * kConsWarps + warp];
      if (__shfl_sync(0xffffffffu, fin, 0)) break;
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
    // ---- park: s_w[warp][head][kPart], once the previous chunk is combined
    if (!wait_gt(&s_misc[18], k - 1)) break;
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
    __syncwarp();
    int last = 0;
    if (lane == 0) {
      __threadfence_block();
      last = atomicAdd(&s_misc[20], 1) == kConsWarps - 1;
      __threadfence_block();
    }
    if (!__shfl_sync(0xffffffffu, last, 0)) continue;
    // ---- the last warp combines the kConsWarps states: lane owns dims [4 lane, 4 lane + 4)
    if (lane == 0) s_misc[20] = 0;
    const bool whole = ci.nch == 1;
    float* part = A.partials + (size_t)(s_cprefix[u * NW] + ci.kin) * PS;
    for (int g = 0; g < G; ++g) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsWarps; ++w) M = fmaxf(M, s_w[(w * G + g) * kPart + kD]);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      float l = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsWarps; ++w) {
          const float* sw = s_w + (w * G + g) * kPart;
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
      if (whole) {
        const size_t row = (size_t)b * p.Hq + kvh * G + g;
        if (p.bypass != nullptr && ((s_umask[u] >> g) & 1)) continue;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        *reinterpret_cast<float4*>(A.out + row * kD + 4 * lane) =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
        if (lane == 0) A.lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
      } else {
        *reinterpret_cast<float4*>(part + g * kD + 4 * lane) = acc;
        if (lane == 0) {
          part[G * kD + g] = M;
          part[G * kD + G + g] = l;
        }
      }
    }
    __syncwarp();
    if (lane == 0) st_release_cta(&s_misc[18], k + 1);   // chunk k combined: s_w and the ring entry are free
  }
}

// ------------------------------------------------------------------ merge

// One CTA per (query head g of the group, unit u): the exact log-sum-exp
// merge of the unit's chunk partials in chunk order; thread d owns dim d.
// Units held in one chunk were finished by the decode kernel.  The decode's
// chunk list is a function of the tile counts and its grid, and the tile
// builder had written the counts before the decode started (so before this
// kernel was launched): the unit's first chunk and chunk count are derived
// before the wait for the decode, and only the partials' loads follow it.
// One pass with a running maximum: the (max, sum, O) loads of kMergeIn
// chunks are issued together, then the running sums are rescaled once to
// the batch's maximum and the batch is added.
constexpr int kMergeThreads = kD;
constexpr int kMergeIn = 16;

__global__ void __launch_bounds__(kMergeThreads)
merge_chunks_kernel(Params p, const float* __restrict__ partials, const int* __restrict__ ntiles, int nwin,
                    int decode_grid, float* __restrict__ out, float* __restrict__ lse) {
  __shared__ int s_red[3][kMergeThreads / 32];
  const int g = blockIdx.x, u = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int SG = p.B * p.Hk * nwin;
  auto block_sum = [&](int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int t = 0;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) t += red[w];
    return t;
  };
  int tsum = 0;
  for (int i = tid; i < SG; i += kMergeThreads) tsum += __ldg(ntiles + i);
  const int T = block_sum(tsum, s_red[0]);   // the decode's chunk size, as it derives it
  const int C = max(kMinChunk, (T + kChunksPerCta * decode_grid - 1) / (kChunksPerCta * decode_grid));
  int before = 0, mine = 0;
  for (int i = tid; i < (u + 1) * nwin; i += kMergeThreads) {
    const int n = (__ldg(ntiles + i) + C - 1) / C;
    if (i < u * nwin) before += n; else mine += n;
  }
  const int c0 = block_sum(before, s_red[1]), nch = block_sum(mine, s_red[2]);
  const size_t row = (size_t)(u / p.Hk) * p.Hq + (u % p.Hk) * p.G + g;
  const bool left_out = p.bypass != nullptr && p.bypass[row];   // complete before the decode started
  pdl_wait();
  pdl_trigger();
  if (nch == 1) return;   // written by the decode; no chunk (nothing attended): O = 0, lse = -inf below
  const int G = p.G, PS = partial_stride(G);
  const float* P = partials + (size_t)c0 * PS;
  float M = -INFINITY, acc = 0.f, l = 0.f;
  for (int j0 = 0; j0 < nch; j0 += kMergeIn) {
    float vm[kMergeIn], vl[kMergeIn], vo[kMergeIn];
#pragma unroll
    for (int t = 0; t < kMergeIn; ++t) {
      if (j0 + t < nch) {
        const float* pc = P + (size_t)(j0 + t) * PS;
        vm[t] = __ldcg(pc + G * kD + g);
        vl[t] = __ldcg(pc + G * kD + G + g);
        vo[t] = __ldcg(pc + g * kD + tid);
      } else {
        vm[t] = -INFINITY;
        vl[t] = 0.f;
        vo[t] = 0.f;
      }
    }
    float Mb = M;
#pragma unroll
    for (int t = 0; t < kMergeIn; ++t) Mb = fmaxf(Mb, vm[t]);
    if (Mb == -INFINITY) continue;
    const float r = M == -INFINITY ? 0.f : exp2f(M - Mb);
    acc *= r;
    l *= r;
#pragma unroll
    for (int t = 0; t < kMergeIn; ++t) {
      const float w = vm[t] == -INFINITY ? 0.f : exp2f(vm[t] - Mb);
      acc += w * vo[t];
      l += w * vl[t];
    }
    M = Mb;
  }
  if (left_out) return;
  out[row * kD + tid] = l > 0.f ? acc / l : 0.f;
  if (tid == 0) lse[row] = l > 0.f ? (M + log2f(l)) * 0.6931471805599453f : -INFINITY;
}

// SG: tile-list segments (units x windows); the bypass mask takes SG >= U bytes.
size_t decode_smem_bytes_n(int SG, int G, int nslots) {
  return 1024 + (size_t)nslots * kTileBytes + kConsWarps * 512 + (size_t)kConsWarps * G * kPart * 4 +
         nslots * sizeof(SlotInfo) + kChunkRing * sizeof(ChunkInfo) + kChunkRing * kConsWarps * 4 +
         2 * nslots * 8 + 32 * 4 +
         (2 * (size_t)(SG + 1) + (SG + 3) / 4) * 4;
}

// Slot count: the largest multiple of kConsWarps (<= 16) that still lets two
// CTAs share an SM; at least kConsWarps.
int decode_slots(int SG, int G) {
  const size_t per_sm = 228 * 1024, reserve = 1024;
  int best = kConsWarps;
  for (int n = kConsWarps; n <= 16; n += kConsWarps)
    if (2 * (decode_smem_bytes_n(SG, G, n) + reserve) <= per_sm) best = n;
  return best;
}

// smallest shared-memory request of the decode for the problem (its fewest slots)
size_t decode_smem_bytes(const Params& p) {
  return decode_smem_bytes_n(p.B * p.Hk * num_windows(p.mpp), kMaxG, kConsWarps);
}

// Chunks never exceed kChunksPerCta * grid + (segments) (the chunk size grows
// with the total beyond kMinChunk tiles per chunk), and the grid never
// exceeds kMaxCtas.
size_t decode_partials_bytes(const Params& p) {
  return ((size_t)kChunksPerCta * kMaxCtas + (size_t)p.B * p.Hk * num_windows(p.mpp)) * partial_stride(p.G) *
         sizeof(float);
}

size_t ntiles_bytes(const Params& p) { return (size_t)p.B * p.Hk * num_windows(p.mpp) * sizeof(int); }

size_t tiles_bytes(const Params& p) { return (size_t)p.B * p.Hk * p.mpp * sizeof(Tile); }

int launch_build_tiles(const Params& p, const int* seq_lens, const int* page_table, const int* sel_idx,
                       const int* sel_cnt, int gran, void* tiles, int* ntiles, int* status, int* ticket,
                       cudaStream_t stream) {
  const size_t smem = build_smem_bytes(p.mpp);
  // static + dynamic shared memory can pass the 48 KB default even when the
  // dynamic part alone does not: always opt in (cached per kernel)
  smem_limit_at_least(reinterpret_cast<const void*>(build_tiles_kernel), (int)smem);
  dim3 grid(p.Hk, p.B, num_windows(p.mpp));   // one CTA per window of each unit
  const cudaError_t e = launch_pdl(build_tiles_kernel, grid, dim3(kBuildThreads), smem, stream, p, seq_lens,
                                   page_table, sel_idx, sel_cnt, gran, static_cast<Tile*>(tiles), ntiles, status,
                                   ticket);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

int launch_decode(const Params& p, const void* q, const int* page_table, const void* tiles, const int* ntiles,
                  float* partials, int* ticket, float* out, float* lse, float* logits, int* status,
                  const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms, cudaStream_t stream) {
  const int U = p.B * p.Hk;
  const int SG = U * num_windows(p.mpp);
  const int nslots = decode_slots(SG, p.G);
  const size_t smem = decode_smem_bytes_n(SG, p.G, nslots);
  if (smem > 227 * 1024) return SA_ERR_UNSUPPORTED;
  void (*kern)(Params, DecodeArgs, const CUtensorMap, const CUtensorMap, int) =
      logits != nullptr ? decode_kernel<true> : decode_kernel<false>;
  smem_limit_at_least(reinterpret_cast<const void*>(kern), (int)smem);
  const int per_sm = ctas_per_sm(reinterpret_cast<const void*>(kern), kDecThreads, smem);
  const int grid = std::min(kMaxCtas, num_sms * per_sm);
  DecodeArgs A;
  A.q = static_cast<const __nv_bfloat16*>(q);
  A.page_table = page_table;
  A.tiles = static_cast<const Tile*>(tiles);
  A.ntiles = ntiles;
  A.partials = partials;
  A.nwin = num_windows(p.mpp);
  A.ticket = ticket;
  A.out = out;
  A.lse = lse;
  A.logits = logits;
  A.status = status;
  cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kDecThreads), smem, stream, p, A, tmK, tmV, nslots);
  if (e != cudaSuccess) return SA_ERR_CUDA;
  e = launch_pdl(merge_chunks_kernel, dim3(p.G, U), dim3(kMergeThreads), 0, stream, p,
                 static_cast<const float*>(partials), ntiles, A.nwin, grid, out, lse);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
