// Exact top-k inside the score-table candidates.
//
// LFPS ("Learn from the Past", "The reading") notes that an exact top-k needs
// a dot product against every key; its tables narrow the keys to a small
// candidate set, and the exact scores are then taken over that set only.
// Here each candidate token's score is q . k_t in the canonical fp32 order
// the block scores use (8 lanes of 16 consecutive dims, ascending, a
// butterfly over lane partners 4, 2, 1, then + 0.0), with the bf16 key row as
// the operand, so the kept set is reproducible bit for bit; the k best by
// (score descending, position ascending) are kept, reported ascending.
//
// One CTA per (query head, sequence).  The candidate positions go to shared
// memory; each warp scores 4 candidates at a time (8 lanes per candidate,
// each lane 32 bytes of the 256-byte key row, found through the page table);
// the scores stay in shared memory for the radix top-k, whose output indices
// are mapped back to positions (a list of at most 32 is ranked by one warp).
#include <algorithm>

#include "sa_common.cuh"
#include "topk.cuh"

namespace sa {

template <int NT, int KPT>
__global__ void __launch_bounds__(NT)
token_topk_kernel(Params p, const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k_pool,
                  const int* __restrict__ page_table, const int* __restrict__ seq_lens,
                  const int* __restrict__ cand_idx, const int* __restrict__ cand_cnt, int* __restrict__ sel_idx,
                  int* __restrict__ sel_cnt, float* __restrict__ scores_out, int* status) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float s_sc[];                 // [kcap] candidate scores, then [kcap] positions
  int* s_cand = reinterpret_cast<int*>(s_sc + p.kcap);
  __shared__ TopkScratch S;
  const int h = blockIdx.x, b = blockIdx.y, kvh = h / p.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = min(seq_lens[b], p.mpp * kP);
  const size_t row = (size_t)b * p.Hq + h;
  const int n = max(0, min(cand_cnt[row], p.kcap));
  for (int e = tid; e < n; e += NT) s_cand[e] = cand_idx[row * p.kcap + e];
  const int sub = lane >> 3, part = lane & 7;     // candidate within the warp's 4, dims [16 part, 16 part + 16)
  uint32_t qw[8];
  {
    const uint4* qr = reinterpret_cast<const uint4*>(q + row * kD) + 2 * part;
    const uint4 a = __ldg(qr), c = __ldg(qr + 1);
    qw[0] = a.x; qw[1] = a.y; qw[2] = a.z; qw[3] = a.w;
    qw[4] = c.x; qw[5] = c.y; qw[6] = c.z; qw[7] = c.w;
  }
  __syncthreads();
  const int* pt = page_table + (size_t)b * p.mpp;
  for (int e0 = warp * 4; e0 < n; e0 += (NT / 32) * 4) {
    const int e = e0 + sub;
    const bool valid = e < n;
    const int t = valid ? s_cand[e] : 0;
    bool in_range = valid && t >= 0 && t < L;     // other entries rank last
    uint4 k0 = make_uint4(0, 0, 0, 0), k1 = make_uint4(0, 0, 0, 0);
    if (in_range) {
      const int phys = __ldg(pt + t / kP);
      if (phys >= 0 && phys < p.num_pages) {
        const uint4* kr =
            reinterpret_cast<const uint4*>(k_pool + (((size_t)phys * p.Hk + kvh) * kP + t % kP) * kD) + 2 * part;
        k0 = __ldg(kr);
        k1 = __ldg(kr + 1);
      } else {
        if (part == 0) set_status(status, SA_ERR_BAD_PAGE);
        in_range = false;
      }
    }
    const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    float acc = 0.f;
#pragma unroll
    for (int k2 = 0; k2 < 8; ++k2) {
      // fma with c = -0 is the plain product, zero signs included
      acc = fma_bf16_lo(qw[k2], kw[k2], k2 == 0 ? -0.0f : acc);
      acc = fma_bf16_hi(qw[k2], kw[k2], acc);
    }
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 4));
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 2));
    acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, 1));
    if (valid && part == 0) s_sc[e] = in_range ? __fadd_rn(acc, 0.0f) : -INFINITY;
  }
  __syncthreads();
  if (scores_out != nullptr)
    for (int e = tid; e < n; e += NT) scores_out[row * p.kcap + e] = s_sc[e];
  int* out = sel_idx + row * p.kcap;
  if (n <= 32) {
    // a short list: warp 0 ranks it directly; a candidate is kept when fewer
    // than k others beat it (higher score, or equal score and lower position)
    if (warp == 0) {
      const uint32_t key = lane < n ? order_key(s_sc[lane]) : 0u;
      int beaten = 0;
      for (int j = 0; j < n; ++j) {
        const uint32_t o = __shfl_sync(0xffffffffu, key, j);
        beaten += (o > key) || (o == key && j < lane);
      }
      const bool keep = lane < n && beaten < p.k[h];
      const unsigned km = __ballot_sync(0xffffffffu, keep);
      if (keep) out[__popc(km & ((1u << lane) - 1u))] = s_cand[lane];
      if (lane == 0) sel_cnt[row] = __popc(km);
    }
    return;
  }
  group_topk<NT, KPT>(s_sc, n, p.k[h], 0, out, sel_cnt + row, 0, S);
  __syncthreads();
  const int m = min(p.k[h], n);
  for (int j = tid; j < m; j += NT) out[j] = s_cand[out[j]];   // indices ascending -> positions ascending
}

size_t token_topk_smem_bytes(const Params& p) { return (size_t)2 * p.kcap * sizeof(float); }

int launch_token_topk(const Params& p, const void* q, const void* k_pool, const int* page_table, const int* seq_lens,
                      const int* cand_idx, const int* cand_cnt, int* sel_idx, int* sel_cnt, float* scores_out,
                      int* status, cudaStream_t stream) {
  const size_t smem = token_topk_smem_bytes(p);
  if (smem > 200 * 1024) return SA_ERR_UNSUPPORTED;
  dim3 grid(p.Hq, p.B);
  const auto* qb = static_cast<const __nv_bfloat16*>(q);
  const auto* kb = static_cast<const __nv_bfloat16*>(k_pool);
  void (*kern)(Params, const __nv_bfloat16*, const __nv_bfloat16*, const int*, const int*, const int*, const int*,
               int*, int*, float*, int*) = nullptr;
  int nt = 0;
  if (p.kcap <= 256 * 8) {
    kern = token_topk_kernel<256, 8>;
    nt = 256;
  } else if (p.kcap <= 1024 * 16) {
    kern = token_topk_kernel<1024, 16>;
    nt = 1024;
  } else if (p.kcap <= 1024 * 64) {
    kern = token_topk_kernel<1024, 64>;
    nt = 1024;
  } else {
    return SA_ERR_UNSUPPORTED;
  }
  smem_limit_at_least(reinterpret_cast<const void*>(kern), (int)smem);
  const cudaError_t e = launch_pdl(kern, grid, dim3(nt), smem, stream, p, qb, kb, page_table, seq_lens, cand_idx,
                                   cand_cnt, sel_idx, sel_cnt, scores_out, status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
