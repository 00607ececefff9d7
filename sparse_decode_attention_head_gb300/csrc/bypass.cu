// Head-sparsity estimate and mean-value bypass (LFPS, "Learn from the Past:
// Fast Sparse Indexing for Large Language Model Decoding": Algorithm 1 step 1,
// Eq. (5), Eq. (6), App. B.1, epsilon = 0.85).
//
// Per (sequence, KV head) the cache keeps running fp32 sums over its L tokens:
// sum k, sum k*k and sum v, per dimension ([B][Hk][3][D]).  For a query head
// with logits z_t = scale q . k_t the estimate splits the tokens into the sink
// (token 0), the local window (the six newest tokens) and the n = L - 7
// global tokens between, and weighs them by
//   sink   e^{z_0}
//   local  sum of e^{z_t} over the window
//   global n exp(scale q . Kbar + scale^2 |q|^2 sigma^2 / 2)
// -- the mean of e^z for keys with independent normal components of mean
// Kbar and variance sigma^2 (the mean over dims of the global keys' per-dim
// variance), which the running sums give after the sink and window rows are
// taken out.  rho = sink / total; rho > epsilon bypasses the head: its output
// is the mean value row over the L tokens and its lse the log of the total.
//
// kv_stats_kernel builds the sums from the cache (one pass, fixed order);
// sparsity_kernel estimates every query head of a KV head with one warp
// (estimate_unit_warp, which the decode step runs in a warp of its score
// kernel).
#include "sa_common.cuh"
#include "sparsity.cuh"

namespace sa {

constexpr int kStatWarps = 16;
constexpr int kStatUnroll = 4;

// One CTA per (KV head, sequence): warp w sums tokens w, w + 16, ... (four in
// flight), lane l dims [4 l, 4 l + 4); the 16 warp partials are then added in
// warp order, so the result does not depend on scheduling.
__global__ void __launch_bounds__(kStatWarps * 32)
kv_stats_kernel(Params p, const __nv_bfloat16* __restrict__ k_pool, const __nv_bfloat16* __restrict__ v_pool,
                const int* __restrict__ page_table, const int* __restrict__ seq_lens, float* __restrict__ stats,
                int* status) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_part[kStatWarps][3 * kD];
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = max(0, min(seq_lens[b], p.mpp * kP));
  const int* pt = page_table + (size_t)b * p.mpp;
  float sk[4] = {0.f, 0.f, 0.f, 0.f}, sq[4] = {0.f, 0.f, 0.f, 0.f}, sv[4] = {0.f, 0.f, 0.f, 0.f};
  bool bad = false;
  for (int t0 = warp; t0 < L; t0 += kStatWarps * kStatUnroll) {
    uint2 kr[kStatUnroll], vr[kStatUnroll];
    bool ok[kStatUnroll];
#pragma unroll
    for (int u = 0; u < kStatUnroll; ++u) {
      const int t = t0 + u * kStatWarps;
      ok[u] = false;
      kr[u] = vr[u] = make_uint2(0u, 0u);
      if (t < L) {
        const int phys = __ldg(pt + t / kP);
        if (phys >= 0 && phys < p.num_pages) {
          const size_t off = (((size_t)phys * p.Hk + kvh) * kP + t % kP) * kD;
          kr[u] = __ldg(reinterpret_cast<const uint2*>(k_pool + off) + lane);
          vr[u] = __ldg(reinterpret_cast<const uint2*>(v_pool + off) + lane);
          ok[u] = true;
        } else {
          bad = true;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kStatUnroll; ++u) {
      if (!ok[u]) continue;
      const float k4[4] = {bf16_lo(kr[u].x), bf16_hi(kr[u].x), bf16_lo(kr[u].y), bf16_hi(kr[u].y)};
      const float v4[4] = {bf16_lo(vr[u].x), bf16_hi(vr[u].x), bf16_lo(vr[u].y), bf16_hi(vr[u].y)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sk[i] += k4[i];
        sq[i] = __fmaf_rn(k4[i], k4[i], sq[i]);
        sv[i] += v4[i];
      }
    }
  }
  if (bad && lane == 0) set_status(status, SA_ERR_BAD_PAGE);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s_part[warp][4 * lane + i] = sk[i];
    s_part[warp][kD + 4 * lane + i] = sq[i];
    s_part[warp][2 * kD + 4 * lane + i] = sv[i];
  }
  __syncthreads();
  float* dst = stats + ((size_t)b * p.Hk + kvh) * 3 * kD;
  for (int i = threadIdx.x; i < 3 * kD; i += kStatWarps * 32) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kStatWarps; ++w) s += s_part[w][i];
    dst[i] = s;
  }
}

int launch_kv_stats(const Params& p, const void* k_pool, const void* v_pool, const int* page_table,
                    const int* seq_lens, float* stats, int* status, cudaStream_t stream) {
  const cudaError_t e =
      launch_pdl(kv_stats_kernel, dim3(p.Hk, p.B), dim3(kStatWarps * 32), 0, stream, p,
                 static_cast<const __nv_bfloat16*>(k_pool), static_cast<const __nv_bfloat16*>(v_pool), page_table,
                 seq_lens, stats, status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

// sa_head_sparsity: one warp per (KV head, sequence).
__global__ void __launch_bounds__(32)
sparsity_kernel(Params p, const __nv_bfloat16* __restrict__ q, const int* __restrict__ seq_lens, EstArgs E) {
  pdl_wait();
  pdl_trigger();
  estimate_unit_warp(p, E, q, seq_lens, blockIdx.y, blockIdx.x);
}

int launch_sparsity(const Params& p, const void* q, const int* seq_lens, const EstArgs& E, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(sparsity_kernel, dim3(p.Hk, p.B), dim3(32), 0, stream, p,
                                   static_cast<const __nv_bfloat16*>(q), seq_lens, E);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
