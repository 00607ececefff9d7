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
// sparsity_kernel optionally appends the new token's rows first (and adds
// them to the sums), then estimates every query head of its KV head.
#include "sa_common.cuh"
#include "summary.cuh"

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

constexpr int kLocalWindow = 6;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// One CTA of 32 G threads per (KV head, sequence).  With k_new, warp 0 first
// writes the new token's rows at L - 1 and adds them to the running sums; the
// block barrier then makes them visible to every head's warp.  Rows written
// here are read back with plain loads.
__global__ void __launch_bounds__(32 * SA_MAX_GROUP)
sparsity_kernel(Params p, const __nv_bfloat16* __restrict__ q, __nv_bfloat16* k_pool, __nv_bfloat16* v_pool,
                const int* __restrict__ page_table, const int* __restrict__ seq_lens,
                const __nv_bfloat16* __restrict__ k_new, const __nv_bfloat16* __restrict__ v_new, float* stats,
                float eps, float* __restrict__ rho_out, int* __restrict__ bypass, float* __restrict__ out,
                float* __restrict__ lse, int* status) {
  pdl_wait();
  pdl_trigger();
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = max(0, min(seq_lens[b], p.mpp * kP));
  const int* pt = page_table + (size_t)b * p.mpp;
  float* st = stats + ((size_t)b * p.Hk + kvh) * 3 * kD;
  if (k_new != nullptr) {
    if (warp == 0 && L > 0) {
      append_token_warp(p, b, kvh, L, k_new, v_new, k_pool, v_pool, pt, status);
      const size_t src = ((size_t)b * p.Hk + kvh) * kD;
      const uint2 kr = reinterpret_cast<const uint2*>(k_new + src)[lane];
      const uint2 vr = reinterpret_cast<const uint2*>(v_new + src)[lane];
      const float k4[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
      const float v4[4] = {bf16_lo(vr.x), bf16_hi(vr.x), bf16_lo(vr.y), bf16_hi(vr.y)};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        st[4 * lane + i] += k4[i];
        st[kD + 4 * lane + i] = __fmaf_rn(k4[i], k4[i], st[kD + 4 * lane + i]);
        st[2 * kD + 4 * lane + i] += v4[i];
      }
    }
    __syncthreads();
  }
  if (warp >= p.G) return;
  const size_t row = (size_t)b * p.Hq + kvh * p.G + warp;
  if (L == 0) {   // nothing to estimate: never bypassed
    if (lane == 0) {
      if (rho_out) rho_out[row] = 0.f;
      bypass[row] = 0;
    }
    return;
  }
  float q4[4];
  {
    const uint2 qr = __ldg(reinterpret_cast<const uint2*>(q + row * kD) + lane);
    q4[0] = bf16_lo(qr.x);
    q4[1] = bf16_hi(qr.x);
    q4[2] = bf16_lo(qr.y);
    q4[3] = bf16_hi(qr.y);
  }
  const float scale = p.scale;
  // the sink and the local window: their logits, and their key sums to take
  // out of the running sums
  const int lo = max(1, L - kLocalWindow);
  float z[1 + kLocalWindow];
  float ek[4] = {0.f, 0.f, 0.f, 0.f}, eq[4] = {0.f, 0.f, 0.f, 0.f};
  bool bad = false;
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) {
    const int t = i == 0 ? 0 : lo + i - 1;
    z[i] = -INFINITY;
    if (i > 0 && t >= L) continue;
    const int phys = pt[t / kP];
    if (phys < 0 || phys >= p.num_pages) {
      bad = true;
      continue;
    }
    const uint2 kr = reinterpret_cast<const uint2*>(k_pool + (((size_t)phys * p.Hk + kvh) * kP + t % kP) * kD)[lane];
    const float k4[4] = {bf16_lo(kr.x), bf16_hi(kr.x), bf16_lo(kr.y), bf16_hi(kr.y)};
    float d = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      d = __fmaf_rn(q4[c], k4[c], d);
      ek[c] += k4[c];
      eq[c] = __fmaf_rn(k4[c], k4[c], eq[c]);
    }
    z[i] = scale * warp_sum(d);
  }
  if (bad) {   // a broken page table: report, never bypass
    if (lane == 0) {
      set_status(status, SA_ERR_BAD_PAGE);
      if (rho_out) rho_out[row] = 0.f;
      bypass[row] = 0;
    }
    return;
  }
  const int n = lo - 1;   // global tokens [1, lo)
  float zg = -INFINITY;
  if (n > 0) {
    const float inv_n = 1.0f / (float)n;
    float qk = 0.f, qq = 0.f, var = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float kbar = (st[4 * lane + c] - ek[c]) * inv_n;
      const float m2 = (st[kD + 4 * lane + c] - eq[c]) * inv_n;
      qk = __fmaf_rn(q4[c], kbar, qk);
      qq = __fmaf_rn(q4[c], q4[c], qq);
      var += fmaxf(0.f, m2 - kbar * kbar);
    }
    qk = warp_sum(qk);
    qq = warp_sum(qq);
    var = warp_sum(var) * (1.0f / kD);
    zg = logf((float)n) + scale * qk + 0.5f * scale * scale * qq * var;
  }
  float m = zg;
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) m = fmaxf(m, z[i]);
  float tot = zg == -INFINITY ? 0.f : expf(zg - m);
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) tot += z[i] == -INFINITY ? 0.f : expf(z[i] - m);
  const float rho = expf(z[0] - m) / tot;
  const bool by = rho > eps;
  if (lane == 0) {
    if (rho_out) rho_out[row] = rho;
    bypass[row] = by ? 1 : 0;
  }
  if (by) {
    const float inv_l = 1.0f / (float)L;
    const float4 o = make_float4(st[2 * kD + 4 * lane] * inv_l, st[2 * kD + 4 * lane + 1] * inv_l,
                                 st[2 * kD + 4 * lane + 2] * inv_l, st[2 * kD + 4 * lane + 3] * inv_l);
    *reinterpret_cast<float4*>(out + row * kD + 4 * lane) = o;
    if (lane == 0) lse[row] = m + logf(tot);
  }
}

int launch_sparsity(const Params& p, const void* q, void* k_pool, void* v_pool, const int* page_table,
                    const int* seq_lens, const void* k_new, const void* v_new, float* stats, float eps, float* rho,
                    int* bypass, float* out, float* lse, int* status, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(
      sparsity_kernel, dim3(p.Hk, p.B), dim3(32 * p.G), 0, stream, p, static_cast<const __nv_bfloat16*>(q),
      static_cast<__nv_bfloat16*>(k_pool), static_cast<__nv_bfloat16*>(v_pool), page_table, seq_lens,
      static_cast<const __nv_bfloat16*>(k_new), static_cast<const __nv_bfloat16*>(v_new), stats, eps, rho, bypass,
      out, lse, status);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
