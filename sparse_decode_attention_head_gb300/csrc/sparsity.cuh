// Head-sparsity estimate of one (sequence, KV head) unit by one warp (LFPS,
// "Learn from the Past: Fast Sparse Indexing for Large Language Model
// Decoding": Algorithm 1 step 1, Eq. (5), Eq. (6), App. B.1).
//
// For each query head of the unit, with logits z_t = scale q . k_t: the sink
// mass e^{z_0}, the local mass (the six newest tokens [max(1, L - 6), L)) and
// the global mass n exp(scale q . Kbar + scale^2 |q|^2 sigma^2 / 2) of the
// n = L - 7 tokens between -- the mean of e^z for keys with independent
// normal components, Kbar their mean and sigma^2 the mean over dims of their
// per-dim variance, taken from the unit's running sums (sum k, sum k*k,
// sum v over the L tokens) minus the sink and window rows.  rho = sink /
// total; rho > eps bypasses the head: out = sum v / L, lse = log total.
//
// Lane l owns dims [4 l, 4 l + 4).  Every global load (page entries, the
// sums, the new token's rows, the heads' q, then the seven key rows) is
// issued before any arithmetic; a head's nine warp sums share one butterfly.
#pragma once

#include "sa_common.cuh"

namespace sa {

constexpr int kLocalWindow = 6;

struct EstArgs {
  const __nv_bfloat16* k_pool;
  const int* page_table;
  // with v_new: the new token's rows, at L - 1 but not yet in the pool when
  // the estimate runs; they are read from here and added to the sums
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  float* stats;   // [B][Hk][3][D]; NULL: no estimate
  float eps;
  float* rho;     // [B][Hq] or NULL
  int* bypass;    // [B][Hq]
  float* out;     // [B][Hq][D]: the mean value row of a bypassed head
  float* lse;     // [B][Hq]
  int* status;
};

__device__ __forceinline__ void unpack4(uint2 w, float (&x)[4]) {
  x[0] = bf16_lo(w.x);
  x[1] = bf16_hi(w.x);
  x[2] = bf16_lo(w.y);
  x[3] = bf16_hi(w.y);
}

// Collective over one warp: every query head of unit (b, kvh).  Pool rows
// are read with plain loads (an earlier kernel of the step may have written
// them).  The sums are only read: with k_new they are taken as the stored
// sums plus the new rows, which the append adds to the stored sums later.
__device__ __forceinline__ void estimate_unit_warp(const Params& p, const EstArgs& E, const __nv_bfloat16* q,
                                                   const int* seq_lens, int b, int kvh) {
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int L = max(0, min(seq_lens[b], p.mpp * kP));
  const size_t row0 = (size_t)b * p.Hq + kvh * G;
  if (L == 0) {   // nothing to estimate: never bypassed
    if (lane < G) {
      if (E.rho) E.rho[row0 + lane] = 0.f;
      E.bypass[row0 + lane] = 0;
    }
    return;
  }
  const int* pt = E.page_table + (size_t)b * p.mpp;
  const bool app = E.k_new != nullptr;
  const int lo = max(1, L - kLocalWindow);
  // ---- loads: page entries, sums, new rows, the heads' q
  int tok[1 + kLocalWindow], phys[1 + kLocalWindow];
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) {
    tok[i] = i == 0 ? 0 : lo + i - 1;
    const bool in_pool = (i == 0 || tok[i] < L) && !(app && tok[i] == L - 1);
    phys[i] = in_pool ? pt[tok[i] / kP] : -1;
  }
  const float4* st = reinterpret_cast<const float4*>(E.stats + ((size_t)b * p.Hk + kvh) * 3 * kD);
  float4 sk = st[lane], sq = st[kD / 4 + lane], sv = st[kD / 2 + lane];
  uint2 nk = make_uint2(0u, 0u), nv = make_uint2(0u, 0u);
  if (app) {
    const size_t src = ((size_t)b * p.Hk + kvh) * kD;
    nk = reinterpret_cast<const uint2*>(E.k_new + src)[lane];
    nv = reinterpret_cast<const uint2*>(E.v_new + src)[lane];
  }
  uint2 qr[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g)
    qr[g] = g < G ? __ldg(reinterpret_cast<const uint2*>(q + (row0 + g) * kD) + lane) : make_uint2(0u, 0u);
  // ---- the sink and window key rows
  uint2 kr[1 + kLocalWindow];
  bool have[1 + kLocalWindow];
  bool bad = false;
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) {
    have[i] = i == 0 || tok[i] < L;
    kr[i] = make_uint2(0u, 0u);
    if (!have[i]) continue;
    if (app && tok[i] == L - 1) {
      kr[i] = nk;
    } else if (phys[i] >= 0 && phys[i] < p.num_pages) {
      kr[i] = reinterpret_cast<const uint2*>(E.k_pool + (((size_t)phys[i] * p.Hk + kvh) * kP + tok[i] % kP) * kD)[lane];
    } else {
      bad = true;
      have[i] = false;
    }
  }
  if (__any_sync(0xffffffffu, bad)) {   // a broken page table: report, never bypass
    if (lane == 0) set_status(E.status, SA_ERR_BAD_PAGE);
    if (lane < G) {
      if (E.rho) E.rho[row0 + lane] = 0.f;
      E.bypass[row0 + lane] = 0;
    }
    return;
  }
  // ---- the sums over all L tokens, then the global tokens' mean and mean
  //      per-dim variance (the sink and window rows taken out)
  if (app) {
    float k4[4], v4[4];
    unpack4(nk, k4);
    unpack4(nv, v4);
    sk.x += k4[0]; sk.y += k4[1]; sk.z += k4[2]; sk.w += k4[3];
    sq.x = __fmaf_rn(k4[0], k4[0], sq.x);
    sq.y = __fmaf_rn(k4[1], k4[1], sq.y);
    sq.z = __fmaf_rn(k4[2], k4[2], sq.z);
    sq.w = __fmaf_rn(k4[3], k4[3], sq.w);
    sv.x += v4[0]; sv.y += v4[1]; sv.z += v4[2]; sv.w += v4[3];
  }
  float kw[1 + kLocalWindow][4];
  float ek[4] = {0.f, 0.f, 0.f, 0.f}, eq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i <= kLocalWindow; ++i) {
    unpack4(kr[i], kw[i]);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (have[i]) {
        ek[c] += kw[i][c];
        eq[c] = __fmaf_rn(kw[i][c], kw[i][c], eq[c]);
      }
  }
  const int n = lo - 1;   // global tokens [1, lo)
  const float inv_n = n > 0 ? 1.0f / (float)n : 0.f;
  const float s1[4] = {sk.x, sk.y, sk.z, sk.w}, s2[4] = {sq.x, sq.y, sq.z, sq.w};
  float kbar[4], var = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    kbar[c] = (s1[c] - ek[c]) * inv_n;
    var += fmaxf(0.f, (s2[c] - eq[c]) * inv_n - kbar[c] * kbar[c]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) var += __shfl_xor_sync(0xffffffffu, var, o);
  const float vmean = var * (1.0f / kD);
  const float scale = p.scale;
  const float inv_l = 1.0f / (float)L;
  const float4 vbar = make_float4(sv.x * inv_l, sv.y * inv_l, sv.z * inv_l, sv.w * inv_l);
  // ---- each query head: the seven logits, q . Kbar and |q|^2, reduced in
  //      one butterfly (independent shuffles in flight)
#pragma unroll 1
  for (int g = 0; g < G; ++g) {
    uint2 qg = qr[0];
#pragma unroll
    for (int e = 1; e < kMaxG; ++e)
      if (e == g) qg = qr[e];
    float q4[4];
    unpack4(qg, q4);
    float red[kLocalWindow + 3];
#pragma unroll
    for (int i = 0; i <= kLocalWindow; ++i) {
      float d = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) d = __fmaf_rn(q4[c], kw[i][c], d);
      red[i] = d;
    }
    float qk = 0.f, qq = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      qk = __fmaf_rn(q4[c], kbar[c], qk);
      qq = __fmaf_rn(q4[c], q4[c], qq);
    }
    red[kLocalWindow + 1] = qk;
    red[kLocalWindow + 2] = qq;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int i = 0; i < kLocalWindow + 3; ++i) red[i] += __shfl_xor_sync(0xffffffffu, red[i], o);
    float z[1 + kLocalWindow];
#pragma unroll
    for (int i = 0; i <= kLocalWindow; ++i) z[i] = have[i] ? scale * red[i] : -INFINITY;
    const float zg = n > 0 ? logf((float)n) + scale * red[kLocalWindow + 1] +
                                 0.5f * scale * scale * red[kLocalWindow + 2] * vmean
                           : -INFINITY;
    float m = zg;
#pragma unroll
    for (int i = 0; i <= kLocalWindow; ++i) m = fmaxf(m, z[i]);
    float tot = zg == -INFINITY ? 0.f : expf(zg - m);
#pragma unroll
    for (int i = 0; i <= kLocalWindow; ++i) tot += z[i] == -INFINITY ? 0.f : expf(z[i] - m);
    const float rho = expf(z[0] - m) / tot;
    const bool by = rho > E.eps;
    const size_t row = row0 + g;
    if (lane == 0) {
      if (E.rho) E.rho[row] = rho;
      E.bypass[row] = by ? 1 : 0;
    }
    if (by) {
      *reinterpret_cast<float4*>(E.out + row * kD + 4 * lane) = vbar;
      if (lane == 0) E.lse[row] = m + logf(tot);
    }
  }
}

// The running sums take the new token's rows (one warp, lane l dims
// [4 l, 4 l + 4)); run after every estimate of the step has read them.
__device__ __forceinline__ void stats_add_new_warp(const Params& p, float* stats, const __nv_bfloat16* k_new,
                                                   const __nv_bfloat16* v_new, int b, int kvh, int L) {
  if (L <= 0) return;
  const int lane = threadIdx.x & 31;
  const size_t src = ((size_t)b * p.Hk + kvh) * kD;
  float k4[4], v4[4];
  unpack4(reinterpret_cast<const uint2*>(k_new + src)[lane], k4);
  unpack4(reinterpret_cast<const uint2*>(v_new + src)[lane], v4);
  float4* st = reinterpret_cast<float4*>(stats + src * 3);
  float4 sk = st[lane], sq = st[kD / 4 + lane], sv = st[kD / 2 + lane];
  sk.x += k4[0]; sk.y += k4[1]; sk.z += k4[2]; sk.w += k4[3];
  sq.x = __fmaf_rn(k4[0], k4[0], sq.x);
  sq.y = __fmaf_rn(k4[1], k4[1], sq.y);
  sq.z = __fmaf_rn(k4[2], k4[2], sq.z);
  sq.w = __fmaf_rn(k4[3], k4[3], sq.w);
  sv.x += v4[0]; sv.y += v4[1]; sv.z += v4[2]; sv.w += v4[3];
  st[lane] = sk;
  st[kD / 4 + lane] = sq;
  st[kD / 2 + lane] = sv;
}

}  // namespace sa
