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
#include "sa_common.cuh"

namespace sa {

constexpr int kScoreWarps = 8;
constexpr int kScoreIters = 4;                                     // 4 blocks per warp per iteration
constexpr int kScoreBlocksPerCta = kScoreWarps * 4 * kScoreIters;  // 128

template <int G, int MODE>
__global__ void __launch_bounds__(kScoreWarps * 32, (G <= 4 ? 2 : 1))
score_kernel(Params p, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ summ,
             const int* __restrict__ seq_lens, float* __restrict__ scores, int always) {
  // the CTA's candidate summaries are contiguous: one bulk copy stages them
  extern __shared__ __align__(128) uint8_t s_sum[];   // kScoreBlocksPerCta x row bytes
  __shared__ uint64_t s_bar;
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int L = min(seq_lens[b], p.mpp * kP);
  const int Bs = p.bs[kvh];
  int j0, j1;
  candidate_range(L, p.S, p.W, Bs, j0, j1);
  const int ncand = j1 - j0;
  const int cta_first = blockIdx.x * kScoreBlocksPerCta;
  if (cta_first >= ncand) return;
  bool all_dense = true;
#pragma unroll
  for (int g = 0; g < G; ++g) all_dense &= (p.k[kvh * G + g] >= ncand);
  if (all_dense && !always) return;  // every head keeps every candidate: no ranking needed

  constexpr int kRowElems = (MODE == SA_SUMMARY_MINMAX) ? 2 * kD : kD;
  constexpr int kRowBytes = kRowElems * 2;
  const int nb = min(kScoreBlocksPerCta, ncand - cta_first);
  const size_t unit_slot = ((size_t)b * p.Hk + kvh) * p.slots;
  if (threadIdx.x == 0) {
    mbar_init(&s_bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&s_bar, nb * kRowBytes);
    bulk_load_1d(s_sum, summ + (unit_slot + j0 + cta_first) * kRowElems, nb * kRowBytes, &s_bar);
  }

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int sub = lane >> 3;   // block within the warp's group of 4
  const int part = lane & 7;   // dims [16 part, 16 part + 16)

  // q of the G heads, this lane's 16 dims, fp32 (exact from bf16)
  float qf[G][16];
  uint32_t selw[G][8];   // byte-permute selectors: take max where q >= 0, else min
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)b * p.Hq + kvh * G + g) * kD + 16 * part);
    const uint4 a = __ldg(src), c = __ldg(src + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qf[g][2 * i] = bf16_lo(w[i]);
      qf[g][2 * i + 1] = bf16_hi(w[i]);
      const bool p0 = qf[g][2 * i] >= 0.f, p1 = qf[g][2 * i + 1] >= 0.f;
      // result bytes 0,1 from kmax (0,1) or kmin (4,5); bytes 2,3 from kmax (2,3) or kmin (6,7)
      selw[g][i] = (p0 ? 0x10u : 0x54u) | (p1 ? 0x3200u : 0x7600u);
    }
  }
  __syncthreads();   // barrier initialised before anyone waits on it
  if (!mbar_wait_bounded(&s_bar, 0, nullptr)) return;

  // lanes 4..7 of a block read their two 16-byte halves in swapped order, so
  // the 8 lanes of a quarter-warp hit 8 distinct bank groups
  const int hf = (part >> 2) & 1;
  const int warp_first = warp * 4 * kScoreIters;
#pragma unroll
  for (int it = 0; it < kScoreIters; ++it) {
    const int cl = warp_first + it * 4 + sub;     // block within the CTA's chunk
    const bool valid = cl < nb;
    const int c = cta_first + cl;
    const uint4* base = reinterpret_cast<const uint4*>(s_sum + (size_t)(valid ? cl : 0) * kRowBytes) + 2 * part;
    uint32_t xmin[8], xmax[8];
    uint4 lo0, lo1;
    {
      const uint4 f = base[hf], s2 = base[hf ^ 1];
      lo0 = hf ? s2 : f;
      lo1 = hf ? f : s2;
    }
    if (MODE == SA_SUMMARY_MINMAX) {
      const uint4 f = base[kD / 8 + hf], s2 = base[kD / 8 + (hf ^ 1)];
      const uint4 hi0 = hf ? s2 : f, hi1 = hf ? f : s2;
      xmin[0] = lo0.x; xmin[1] = lo0.y; xmin[2] = lo0.z; xmin[3] = lo0.w;
      xmin[4] = lo1.x; xmin[5] = lo1.y; xmin[6] = lo1.z; xmin[7] = lo1.w;
      xmax[0] = hi0.x; xmax[1] = hi0.y; xmax[2] = hi0.z; xmax[3] = hi0.w;
      xmax[4] = hi1.x; xmax[5] = hi1.y; xmax[6] = hi1.z; xmax[7] = hi1.w;
    } else {
      xmax[0] = lo0.x; xmax[1] = lo0.y; xmax[2] = lo0.z; xmax[3] = lo0.w;
      xmax[4] = lo1.x; xmax[5] = lo1.y; xmax[6] = lo1.z; xmax[7] = lo1.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) xmin[i] = 0u;
    }
    float my_score = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t w = (MODE == SA_SUMMARY_MINMAX) ? __byte_perm(xmax[i], xmin[i], selw[g][i]) : xmax[i];
        if (i == 0)
          acc = __fmul_rn(qf[g][0], bf16_lo(w));
        else
          acc = __fmaf_rn(qf[g][2 * i], bf16_lo(w), acc);
        acc = __fmaf_rn(qf[g][2 * i + 1], bf16_hi(w), acc);
      }
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
      acc = __fadd_rn(acc, 0.0f);
      if (part == g) my_score = acc;
    }
    if (valid && part < G) scores[((size_t)b * p.Hq + kvh * G + part) * p.slots + j0 + c] = my_score;
  }
}

// ---------------------------------------------------------------- top-k

constexpr int kTopkThreads = 512;

__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread; returns the prefix and
// writes the total to *total.  Uses `tmp` (>= 32 ints of shared memory).
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) tmp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) tmp[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  const int before = (warp > 0 ? tmp[warp - 1] : 0) + x - v;
  *total = tmp[nw - 1];
  __syncthreads();
  return before;
}

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(Params p, const float* __restrict__ scores, const int* __restrict__ seq_lens,
            int* __restrict__ sel_idx, int* __restrict__ sel_cnt) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[256];
  __shared__ int scan_tmp[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_krem;

  const int h = blockIdx.x, b = blockIdx.y;
  const int kvh = h / p.G;
  const int L = min(seq_lens[b], p.mpp * kP);
  const int Bs = p.bs[kvh];
  int j0, j1;
  candidate_range(L, p.S, p.W, Bs, j0, j1);
  const int n = j1 - j0;
  const int k = min(p.k[h], n);
  int* out = sel_idx + ((size_t)b * p.Hq + h) * p.kcap;
  const int tid = threadIdx.x;

  if (k >= n) {  // keep every candidate (100 % budget, or no candidates); n <= k <= kcap
    for (int i = tid; i < n; i += blockDim.x) out[i] = j0 + i;
    if (tid == 0) sel_cnt[(size_t)b * p.Hq + h] = n;
    return;
  }
  if (k <= 0) {
    if (tid == 0) sel_cnt[(size_t)b * p.Hq + h] = 0;
    return;
  }

  const float* sc = scores + ((size_t)b * p.Hq + h) * p.slots + j0;
  for (int i = tid; i < n; i += blockDim.x) keys[i] = order_key(sc[i]);

  uint32_t prefix = 0, mask = 0;
  int krem = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    // warp-aggregated: one atomic per distinct digit per warp (in the top
    // passes nearly all keys share a digit)
    for (int base = 0; base < n; base += blockDim.x) {
      const int i = base + tid;
      const uint32_t u = i < n ? keys[i] : 0u;
      const bool take = i < n && (u & mask) == prefix;
      const uint32_t digit = (u >> shift) & 255u;
      const unsigned act = __ballot_sync(0xffffffffu, take);
      if (take) {
        const unsigned peers = __match_any_sync(act, digit);
        if ((threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
      }
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns digits 255-8l .. 248-8l (descending)
      int cnt[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) { cnt[i] = hist[255 - 8 * tid - i]; tot += cnt[i]; }
      int incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int above = incl - tot;
      if (above < krem && krem <= incl) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above < krem && krem <= above + cnt[i]) {
            s_prefix = prefix | ((uint32_t)(255 - 8 * tid - i) << shift);
            s_krem = krem - above;
          }
          above += cnt[i];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    krem = s_krem;
    mask |= 255u << shift;
  }
  const uint32_t T = prefix;   // key of the k-th best
  const int need_eq = krem;    // how many keys equal to T are taken (lowest index first)

  // stable compaction in ascending index order
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int eq = 0;
  for (int i = lo; i < hi; ++i) eq += (keys[i] == T);
  int tot;
  const int eq_before = block_excl_scan(eq, scan_tmp, &tot);
  int take = 0;
  {
    int r = eq_before;
    for (int i = lo; i < hi; ++i) {
      const uint32_t u = keys[i];
      if (u > T) ++take;
      else if (u == T) { if (r < need_eq) ++take; ++r; }
    }
  }
  const int pos0 = block_excl_scan(take, scan_tmp, &tot);
  {
    int r = eq_before, pos = pos0;
    for (int i = lo; i < hi; ++i) {
      const uint32_t u = keys[i];
      bool t = false;
      if (u > T) t = true;
      else if (u == T) { t = r < need_eq; ++r; }
      if (t) out[pos++] = j0 + i;
    }
  }
  if (tid == 0) sel_cnt[(size_t)b * p.Hq + h] = k;
}

int launch_score(const Params& p, const void* q, const void* summ, const int* seq_lens, float* scores,
                 int always, cudaStream_t stream) {
  dim3 grid((p.slots + kScoreBlocksPerCta - 1) / kScoreBlocksPerCta, p.Hk, p.B);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* sb = static_cast<const __nv_bfloat16*>(summ);
  const size_t smem_mm = (size_t)kScoreBlocksPerCta * 2 * kD * 2, smem_mean = smem_mm / 2;
#define SA_SCORE_CASE(GG)                                                                          \
  case GG:                                                                                         \
    if (p.mode == SA_SUMMARY_MINMAX) {                                                             \
      cudaFuncSetAttribute(score_kernel<GG, SA_SUMMARY_MINMAX>,                                    \
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_mm);             \
      score_kernel<GG, SA_SUMMARY_MINMAX>                                                          \
          <<<grid, kScoreWarps * 32, smem_mm, stream>>>(p, qb, sb, seq_lens, scores, always);      \
    } else {                                                                                       \
      score_kernel<GG, SA_SUMMARY_MEAN>                                                            \
          <<<grid, kScoreWarps * 32, smem_mean, stream>>>(p, qb, sb, seq_lens, scores, always);    \
    }                                                                                              \
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
#undef SA_SCORE_CASE
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

size_t topk_smem_bytes(const Params& p) { return (size_t)p.slots * sizeof(uint32_t); }

int launch_topk(const Params& p, const float* scores, const int* seq_lens, int* sel_idx, int* sel_cnt,
                cudaStream_t stream) {
  const size_t smem = topk_smem_bytes(p);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(p.Hq, p.B);
  topk_kernel<<<grid, kTopkThreads, smem, stream>>>(p, scores, seq_lens, sel_idx, sel_cnt);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
