// Steps a2 + a3: block scores in the canonical fp32 order, then per-head top-k.
//
// Fluxion (core claim, Fig. 2d) selects a top-k set of KV blocks per head,
// each head with its own block size and budget.  The selection has to be
// reproducible bit for bit, so scores are accumulated in one fixed fp32
// order (no tensor cores: their internal accumulation order is not defined):
//   8 lanes per block, lane l owns dims [16l, 16l+16) and sums its exact
//   bf16 x bf16 products in ascending dim order (one rounding per step), then
//   a butterfly over lane partners at offsets 4, 2, 1, then + 0.0.
// A warp scores 4 blocks at once for all G query heads of the KV head, so
// each summary byte is read from HBM once per group.
//
// Top-k keeps the k best blocks by (score desc, block index asc): a 4-pass
// MSB-first radix select over order-preserving uint32 keys finds the k-th
// key T and how many keys equal to T to take; a stable block-wide
// compaction then emits the chosen indices in ascending order.
#include <algorithm>

#include "sa_common.cuh"
#include "sparsity.cuh"
#include "topk.cuh"

namespace sa {

constexpr int kScoreWarps = 15;                // consumer warps (+1 producer warp: 4 warps per scheduler)
// threads of a CTA: the consumers, the producer, and with EST the warp of the
// head-sparsity estimate
constexpr int score_threads(bool est) { return (kScoreWarps + (est ? 2 : 1)) * 32; }
constexpr int kMaxUnitsScore = 4096;

// Work items are (unit = (b, kv head), run of kItemBlocks candidate blocks).
// Each CTA takes a contiguous range of items; a producer thread streams each
// item's summaries (contiguous) and the group's q into a ring of shared-memory
// stages with 1-D bulk copies, and leaves a descriptor of the item (where its
// scores go, how many blocks it holds) beside the stage; consumer warps score
// the staged blocks.  With EST a last warp runs the head-sparsity estimate of
// units blockIdx.x, blockIdx.x + gridDim.x, ... beside them (its own
// instantiation: the extra warp lowers the register cap).
struct ItemDesc {
  long long sbase;   // scores index of (b, first head of the group, first block of the item)
  int nb;            // blocks in the item
  int unit;          // b * Hk + kvh
};

// Work split for a group of G query heads.  A consumer warp scores 4 blocks
// at a time (8 lanes per block) for a set of up to 4 heads (q is held packed,
// 8 registers per head, plus 8 selector words per head for min/max); the head
// sets of a group of warps cover the G heads of the same 4 blocks, so each
// staged summary byte is read from shared memory once per head set.  An item
// is as many blocks as the consumer warps take in kRounds passes.
template <int G>
struct ScoreShape {
  static constexpr int kPerWarp = G < 4 ? G : 4;
  static constexpr int kSets = (G + kPerWarp - 1) / kPerWarp;
  static constexpr int kGroups = kScoreWarps / kSets;   // 4-block groups per pass
  static constexpr int kRounds = kSets == 1 ? 1 : 2;
  static constexpr int kItemBlocks = 4 * kGroups * kRounds;
};

constexpr int item_blocks(int G) {
  return G == 1 ? ScoreShape<1>::kItemBlocks : G == 2 ? ScoreShape<2>::kItemBlocks
       : G == 3 ? ScoreShape<3>::kItemBlocks : G == 4 ? ScoreShape<4>::kItemBlocks
       : G == 5 ? ScoreShape<5>::kItemBlocks : G == 6 ? ScoreShape<6>::kItemBlocks
       : G == 7 ? ScoreShape<7>::kItemBlocks : ScoreShape<8>::kItemBlocks;
}

template <int G, int MODE, bool EST>
__global__ void __launch_bounds__(score_threads(EST), 1)
score_kernel(Params p, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ summ,
             const int* __restrict__ seq_lens, float* __restrict__ scores, int always, int nstages, EstArgs E) {
  pdl_wait();
  pdl_trigger();
  constexpr int kRowElems = (MODE == SA_SUMMARY_MINMAX) ? 2 * kD : kD;
  constexpr int kRowBytes = kRowElems * 2;
  constexpr int kItemBlocks = ScoreShape<G>::kItemBlocks;
  constexpr int kStageBytes = kItemBlocks * kRowBytes + kMaxG * kD * 2;   // summaries + q
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t s_full[16], s_empty[16];
  __shared__ ItemDesc s_desc[16];
  __shared__ int s_items[kMaxUnitsScore + 1];   // prefix of items over units

  const int U = p.B * p.Hk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // items per unit (0 when every head keeps every candidate and scores are not asked for)
  for (int u = tid; u < U; u += blockDim.x) {
    const int b = u / p.Hk, kvh = u % p.Hk;
    const int L = min(seq_lens[b], p.mpp * kP);
    int j0, j1;
    candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
    const int ncand = j1 - j0;
    bool all_dense = true;
    for (int g = 0; g < G; ++g) all_dense &= (p.k[kvh * G + g] >= ncand);
    s_items[u + 1] = (all_dense && !always) ? 0 : (ncand + kItemBlocks - 1) / kItemBlocks;
  }
  if (tid == 0) {
    for (int i = 0; i < nstages; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kScoreWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == 0) {   // inclusive scan of the item counts, 32 units at a time
    int carry = 0;
    for (int base = 0; base < U; base += 32) {
      const int u = base + lane;
      const int x = warp_incl_scan(u < U ? s_items[u + 1] : 0);
      if (u < U) s_items[u + 1] = x + carry;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) s_items[0] = 0;
  }
  __syncthreads();
  const long long total = s_items[U];
  const long long it_lo = total * blockIdx.x / gridDim.x, it_hi = total * (blockIdx.x + 1) / gridDim.x;
  const int n_items = (int)(it_hi - it_lo);
  if (EST && warp == kScoreWarps + 1) {   // ---------------- head-sparsity estimate
    for (int u = blockIdx.x; u < U; u += gridDim.x) estimate_unit_warp(p, E, q, seq_lens, u / p.Hk, u % p.Hk);
    return;
  }
  if (n_items <= 0) return;

  if (warp == kScoreWarps) {   // ---------------- producer
    if (lane == 0) {
      int lo = 0, hi = U;   // unit holding the first item
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_items[mid] <= it_lo) lo = mid; else hi = mid;
      }
      int u = lo;
      for (int i = 0; i < n_items; ++i) {
        // describe the item before waiting for its stage
        const long long it = it_lo + i;
        while (it >= s_items[u + 1]) ++u;
        const int b = u / p.Hk, kvh = u % p.Hk;
        const int L = min(seq_lens[b], p.mpp * kP);
        int j0, j1;
        candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
        const int first = (int)(it - s_items[u]) * kItemBlocks;
        const int nb = min(kItemBlocks, (j1 - j0) - first);
        const int st = i % nstages, use = i / nstages;
        if (use > 0 && !mbar_wait_bounded(&s_empty[st], (use - 1) & 1, nullptr)) break;
        s_desc[st] = ItemDesc{((long long)b * p.Hq + kvh * G) * p.slots + j0 + first, nb, u};
        uint8_t* dst = smem + (size_t)st * kStageBytes;
        mbar_arrive_expect_tx(&s_full[st], nb * kRowBytes + G * kD * 2);   // release: orders s_desc
        bulk_load_1d(dst, summ + ((((size_t)b * p.Hk + kvh) * p.slots) + j0 + first) * kRowElems, nb * kRowBytes,
                     &s_full[st]);
        bulk_load_1d(dst + kItemBlocks * kRowBytes, q + ((size_t)b * p.Hq + kvh * G) * kD, G * kD * 2, &s_full[st]);
      }
    }
    return;
  }

  // ---------------- consumers
  constexpr int HPW = ScoreShape<G>::kPerWarp;
  constexpr int NS = ScoreShape<G>::kSets;
  constexpr int GROUPS = ScoreShape<G>::kGroups;
  constexpr int ROUNDS = ScoreShape<G>::kRounds;
  const int hset = warp % NS, grp = warp / NS;
  const bool active_warp = grp < GROUPS;
  const int sub = lane >> 3;   // block within the warp's group of 4
  const int part = lane & 7;   // dims [16 part, 16 part + 16)
  uint32_t qw[HPW][8];         // q of the warp's heads, this lane's 16 dims, packed bf16
  uint32_t selw[HPW][8];       // byte selectors: kmax where q >= 0, else kmin
  int cur_unit = -1;
  for (int i = 0; i < n_items; ++i) {
    const int st = i % nstages, use = i / nstages;
    if (!mbar_wait_bounded(&s_full[st], use & 1, nullptr)) break;
    const ItemDesc dsc = s_desc[st];
    const uint8_t* stage = smem + (size_t)st * kStageBytes;
    if (active_warp) {
      if (dsc.unit != cur_unit) {
        cur_unit = dsc.unit;
        const uint4* qs = reinterpret_cast<const uint4*>(stage + kItemBlocks * kRowBytes);
#pragma unroll
        for (int e = 0; e < HPW; ++e) {
          const int g = hset * HPW + e;
          const int gg = g < G ? g : 0;
          const uint4 a = qs[gg * (kD / 8) + 2 * part], c = qs[gg * (kD / 8) + 2 * part + 1];
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2) {
            qw[e][k2] = w[k2];
            const bool p0 = bf16_lo(w[k2]) >= 0.f, p1 = bf16_hi(w[k2]) >= 0.f;
            // result bytes 0,1 from kmax (0,1) or kmin (4,5); bytes 2,3 from kmax (2,3) or kmin (6,7)
            selw[e][k2] = (p0 ? 0x10u : 0x54u) | (p1 ? 0x3200u : 0x7600u);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < ROUNDS; ++r) {
        const int cl = (r * GROUPS + grp) * 4 + sub;   // block within the item
        const bool valid = cl < dsc.nb;
        const uint4* base = reinterpret_cast<const uint4*>(stage + (size_t)(valid ? cl : 0) * kRowBytes) + 2 * part;
        uint32_t xmin[8], xmax[8];
        {
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
        }
        float acc[HPW];
#pragma unroll
        for (int e = 0; e < HPW; ++e) {
          float a = 0.f;
#pragma unroll
          for (int k2 = 0; k2 < 8; ++k2) {
            const uint32_t w = (MODE == SA_SUMMARY_MINMAX) ? __byte_perm(xmax[k2], xmin[k2], selw[e][k2]) : xmax[k2];
            // fma with c = -0 is the plain product, zero signs included
            a = fma_bf16_lo(qw[e][k2], w, k2 == 0 ? -0.0f : a);
            a = fma_bf16_hi(qw[e][k2], w, a);
          }
          acc[e] = a;
        }
        if (HPW == 4) {
          // Butterfly over the parts with the heads spread over the lanes: at
          // partner distance 4 a lane keeps two heads and sends the other
          // two, at distance 2 it keeps one, at distance 1 both partners hold
          // the same head.  Every add is (own partial) + (partner's partial)
          // of one head, the sums of the plain per-head butterfly.
          const bool b2 = (part & 4) != 0, b1 = (part & 2) != 0;
          const float r0 = __shfl_xor_sync(0xffffffffu, b2 ? acc[0] : acc[2], 4);
          const float r1 = __shfl_xor_sync(0xffffffffu, b2 ? acc[1] : acc[3], 4);
          const float x0 = __fadd_rn(b2 ? acc[2] : acc[0], r0);   // head 2 b2
          const float x1 = __fadd_rn(b2 ? acc[3] : acc[1], r1);   // head 2 b2 + 1
          const float r2 = __shfl_xor_sync(0xffffffffu, b1 ? x0 : x1, 2);
          const float y = __fadd_rn(b1 ? x1 : x0, r2);            // head 2 b2 + b1
          const float z = __fadd_rn(y, __shfl_xor_sync(0xffffffffu, y, 1));
          const float v = __fadd_rn(z, 0.0f);
          const int g = hset * HPW + (part >> 1);
          if (valid && (part & 1) == 0 && g < G) scores[dsc.sbase + (long long)g * p.slots + cl] = v;
        } else {
          float res[HPW];
#pragma unroll
          for (int e = 0; e < HPW; ++e) {
            float a = acc[e];
            a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 4));
            a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 2));
            a = __fadd_rn(a, __shfl_xor_sync(0xffffffffu, a, 1));
            res[e] = __fadd_rn(a, 0.0f);
          }
          // lane part e writes head hset * HPW + e
          float v = res[0];
#pragma unroll
          for (int e = 1; e < HPW; ++e)
            if (part == e) v = res[e];
          const int g = hset * HPW + part;
          if (valid && part < HPW && g < G) scores[dsc.sbase + (long long)g * p.slots + cl] = v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[st]);
  }
}

// ---------------------------------------------------------------- top-k

// GRP: group-shared selection, its own instantiation (see select_build_kernel).
template <int NT, int KPT, bool GRP>
__global__ void __launch_bounds__(NT)
topk_kernel(Params p, const float* __restrict__ scores, const int* __restrict__ seq_lens,
            int* __restrict__ sel_idx, int* __restrict__ sel_cnt) {
  pdl_wait();
  pdl_trigger();
  __shared__ TopkScratch S;
  const int b = blockIdx.y;
  const int L = min(seq_lens[b], p.mpp * kP);
  int j0, j1;
  if (GRP) {   // one CTA per KV head: the group's summed scores, one list for all
    const int kvh = blockIdx.x, h0 = kvh * p.G;
    candidate_range(L, p.S, p.W, p.bs[kvh], j0, j1);
    int* row0 = sel_idx + ((size_t)b * p.Hq + h0) * p.kcap;
    group_topk<NT, KPT, true>(scores + ((size_t)b * p.Hq + h0) * p.slots + j0, j1 - j0, p.k[h0], j0, row0,
                              sel_cnt + (size_t)b * p.Hq + h0, 0, S, p.G, (size_t)p.slots);
    __syncthreads();
    const int cnt = sel_cnt[(size_t)b * p.Hq + h0];
    for (int g = 1; g < p.G; ++g) {
      for (int i = threadIdx.x; i < cnt; i += NT) row0[(size_t)g * p.kcap + i] = row0[i];
      if (threadIdx.x == 0) sel_cnt[(size_t)b * p.Hq + h0 + g] = cnt;
    }
    return;
  }
  const int h = blockIdx.x;
  candidate_range(L, p.S, p.W, p.bs[h / p.G], j0, j1);
  group_topk<NT, KPT>(scores + ((size_t)b * p.Hq + h) * p.slots + j0, j1 - j0, p.k[h], j0,
                      sel_idx + ((size_t)b * p.Hq + h) * p.kcap, sel_cnt + (size_t)b * p.Hq + h, 0, S);
}

int launch_score(const Params& p, const void* q, const void* summ, const int* seq_lens, float* scores,
                 int always, int num_sms, cudaStream_t stream, const EstArgs* est_args) {
  if (p.B * p.Hk > kMaxUnitsScore) return SA_ERR_UNSUPPORTED;
  EstArgs E{};
  if (est_args != nullptr) E = *est_args;
  const bool est = E.stats != nullptr;
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* sb = static_cast<const __nv_bfloat16*>(summ);
  const int row_bytes = (p.mode == SA_SUMMARY_MINMAX ? 2 : 1) * kD * 2;
  const size_t stage = (size_t)item_blocks(p.G) * row_bytes + kMaxG * kD * 2;
  const int nstages = (int)std::min<size_t>(16, (200 * 1024) / stage);
  const size_t smem = stage * nstages;
  const int grid = std::max(1, num_sms);
  cudaError_t err = cudaSuccess;
#define SA_SCORE_LAUNCH(GG, MM, EE)                                                       \
  smem_limit_at_least(reinterpret_cast<const void*>(score_kernel<GG, MM, EE>), (int)smem); \
  err = launch_pdl(score_kernel<GG, MM, EE>, dim3(grid), dim3(score_threads(EE)), smem,    \
                   stream, p, qb, sb, seq_lens, scores, always, nstages, E);
#define SA_SCORE_CASE(GG)                                  \
  case GG:                                                 \
    if (p.mode == SA_SUMMARY_MINMAX) {                     \
      if (est) {                                           \
        SA_SCORE_LAUNCH(GG, SA_SUMMARY_MINMAX, true)       \
      } else {                                             \
        SA_SCORE_LAUNCH(GG, SA_SUMMARY_MINMAX, false)      \
      }                                                    \
    } else if (est) {                                      \
      SA_SCORE_LAUNCH(GG, SA_SUMMARY_MEAN, true)           \
    } else {                                               \
      SA_SCORE_LAUNCH(GG, SA_SUMMARY_MEAN, false)          \
    }                                                      \
    break;
  switch (p.G) {
    SA_SCORE_CASE(1)
    SA_SCORE_CASE(2)
    SA_SCORE_CASE(3)
    SA_SCORE_CASE(4)
    SA_SCORE_CASE(5)
    SA_SCORE_CASE(6)
    SA_SCORE_CASE(7)
    SA_SCORE_CASE(8)
    default:
      return SA_ERR_UNSUPPORTED;
  }
#undef SA_SCORE_LAUNCH
#undef SA_SCORE_CASE
  return err == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

size_t topk_smem_bytes(const Params&) { return 0; }

int launch_topk(const Params& p, const float* scores, const int* seq_lens, int* sel_idx, int* sel_cnt,
                cudaStream_t stream) {
  dim3 grid(p.sel_mode == SA_SELECT_GROUP ? p.Hk : p.Hq, p.B);
  const int max_n = max_candidates(p);
  const bool grp = p.sel_mode == SA_SELECT_GROUP;
  cudaError_t e;
  // the smallest CTA that holds every candidate, so that CTAs of many heads share an SM
  if (max_n <= 256 * 8)
    e = launch_pdl(grp ? topk_kernel<256, 8, true> : topk_kernel<256, 8, false>, grid, dim3(256), 0, stream, p,
                   scores, seq_lens, sel_idx, sel_cnt);
  else if (max_n <= 256 * 16)
    e = launch_pdl(grp ? topk_kernel<256, 16, true> : topk_kernel<256, 16, false>, grid, dim3(256), 0, stream, p,
                   scores, seq_lens, sel_idx, sel_cnt);
  else if (max_n <= 512 * 16)
    e = launch_pdl(grp ? topk_kernel<512, 16, true> : topk_kernel<512, 16, false>, grid, dim3(512), 0, stream, p,
                   scores, seq_lens, sel_idx, sel_cnt);
  else if (max_n <= 1024 * 16)
    e = launch_pdl(grp ? topk_kernel<1024, 16, true> : topk_kernel<1024, 16, false>, grid, dim3(1024), 0, stream, p,
                   scores, seq_lens, sel_idx, sel_cnt);
  else if (max_n <= 1024 * 64)
    e = launch_pdl(grp ? topk_kernel<1024, 64, true> : topk_kernel<1024, 64, false>, grid, dim3(1024), 0, stream, p,
                   scores, seq_lens, sel_idx, sel_cnt);
  else
    return SA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
