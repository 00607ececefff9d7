// Step a7: vertical / slash score tables, updated after a decode step and
// thresholded into the next step's candidate tokens, in one pass.
//
// LFPS ("Learn from the Past", "What carries the argument", Eq. (10)) keeps,
// per head, a table indexed by absolute key position (vertical) and one
// indexed by offset from the newest token (slash), decayed by r = 0.95 each
// step and fed with the step's attention weights; HGCA's moving average of
// attention weights is the vertical table and its keep rule is
// "average > beta / (entries attended densely)".  LFPS Eq. (9) expands each
// candidate by offsets {-1, 0, 1, 2}.
//
// Arithmetic (fp32): w = (1 - r) * exp(z - lse) for an attended entry of the
// previous step (z, lse from sa_sparse_decode), 0 otherwise;
// T_new = fma(r, T_old, w).  Candidate test: T_new > beta / |I| in fp32.
//
// One CTA per (chunk of kChunk positions, query head, sequence): it builds
// the chunk's weights in shared memory (dense-set entries directly, selected
// tokens from the sorted previous selection list), updates and writes both
// tables (the slash entry tested at position i is offset L - 1 - i), marks
// seeds (recomputing the 3-position halo its neighbours own), expands them,
// and compacts the chunk's candidates in ascending order into a staging row
// (at most min(kChunk, kcap) kept) with their count.  A second kernel
// concatenates each head's chunks in order into the candidate list.  Tables
// are double-buffered (read in, write out) so no CTA reads an entry another
// has already rewritten.
#include <algorithm>

#include "tables.cuh"

namespace sa {

constexpr int kTabThreads = 512;
constexpr int kPer = 8;                        // positions per thread per chunk
constexpr int kChunk = kTabThreads * kPer;     // 4096
constexpr int kHalo = 3;                       // seeds at i-2 .. i+1 expand onto i


// Weight fed to the tables by an entry the previous step attended:
// (1 - r) e^(z - lse), z its logit.
__device__ __forceinline__ float attended_weight(const float* logits, int pos, float lse, float one_minus_r) {
  return __fmul_rn(one_minus_r, expf(__ldg(logits + pos) - lse));
}

__global__ void __launch_bounds__(kTabThreads)
tables_kernel(Params p, TableArgs A) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_wv[kChunk + kHalo];       // weights feeding the vertical entries (positions c0-2 ..)
  __shared__ float s_ws[kChunk + kHalo];       // weights feeding the slash entries tested there
  // seed bits by position offset o = j - c0, stored at bit o + 32: word 0
  // holds the left halo (o = -2, -1 at bits 30, 31), words 1 .. kChunk / 32
  // the chunk, the word after them the right halo (o = kChunk)
  __shared__ uint32_t s_seed[kChunk / 32 + 2];
  __shared__ int s_scan[32];
  __shared__ int s_total;

  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.mpp * kP;                                  // table length
  const size_t row = ((size_t)b * p.Hq + h) * N;
  const float* vin = A.vin + row;
  const float* sin = A.sin + row;
  float* vout = A.vout + row;
  float* sout = A.sout + row;
  const int L = min(A.lens[b], N);
  int s_end, w_beg;
  partition(L, p.S, p.W, s_end, w_beg);
  const int n_dense = s_end + (L - w_beg);
  const float tau = n_dense > 0 ? __fdiv_rn(A.beta, (float)n_dense) : INFINITY;
  const float r = A.decay, one_minus_r = __fsub_rn(1.0f, A.decay);
  const bool has_prev = A.prev_logits != nullptr && !(A.frozen != nullptr && A.frozen[(size_t)b * p.Hq + h]);
  int Lp = 0, ps_end = 0, pw_beg = 0, scnt = 0;
  float lse = 0.f;
  const int* sel = nullptr;
  const float* logits = nullptr;
  if (has_prev) {
    Lp = min(A.prev_lens[b], N);
    partition(Lp, p.S, p.W, ps_end, pw_beg);
    sel = A.prev_sel + ((size_t)b * p.Hq + h) * p.kcap;
    scnt = max(0, min(A.prev_cnt[(size_t)b * p.Hq + h], p.kcap));
    lse = A.prev_lse[(size_t)b * p.Hq + h];
    logits = A.prev_logits + row;
  }
  const int delta = L - Lp;   // positions the context grew by since the previous step
  const int nch = (N + kChunk - 1) / kChunk;
  const int cap = min(kChunk, p.kcap);
  const int row_id = b * p.Hq + h;
  int* stage = A.stage + ((size_t)row_id * nch + blockIdx.x) * cap;
  const int c0 = blockIdx.x * kChunk;
  const int c1 = min(N, c0 + kChunk);
  const int n = c1 - c0 + kHalo;                             // positions c0-2 .. c1
  const int base_v = c0 - 2, base_s = c0 - 2 - delta;       // previous-step position of entry k

  // 1. this thread's entries, positions c0 + tid + q kTabThreads (so a warp's
  //    loads are contiguous in both tables), loaded first
  float vv[kPer], sv[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int j = c0 + tid + q * kTabThreads;
    const int d = L - 1 - j;                                 // slash offset tested at this position
    vv[q] = j < c1 ? __ldg(vin + j) : 0.f;
    sv[q] = (j < c1 && d >= 0 && d < N) ? __ldg(sin + d) : 0.f;
  }

  // 2. the previous step's weights on the chunk (and its halo), in shared memory
  if (has_prev) {
    for (int k = tid; k < n; k += kTabThreads) {
      s_wv[k] = 0.f;
      s_ws[k] = 0.f;
    }
    __syncthreads();
    // dense-set entries: [0, ps_end) and [pw_beg, Lp)
    auto dense_fill = [&](float* w, int base) {
      for (int pos = max(base, 0) + tid; pos < min(base + n, ps_end); pos += kTabThreads)
        w[pos - base] = attended_weight(logits, pos, lse, one_minus_r);
      for (int pos = max(base, pw_beg) + tid; pos < min(base + n, Lp); pos += kTabThreads)
        w[pos - base] = attended_weight(logits, pos, lse, one_minus_r);
    };
    dense_fill(s_wv, base_v);
    dense_fill(s_ws, base_s);
    // selected entries inside the previous middle region: every thread scans
    // part of the list (duplicates write the same value)
    for (int e = tid; e < scnt; e += kTabThreads) {
      const int pos = __ldg(sel + e);
      if (pos < ps_end || pos >= pw_beg) continue;
      const int kv = pos - base_v, ks = pos - base_s;
      const bool inv = kv >= 0 && kv < n, ins = ks >= 0 && ks < n;
      if (!inv && !ins) continue;
      const float wt = attended_weight(logits, pos, lse, one_minus_r);
      if (inv) s_wv[kv] = wt;
      if (ins) s_ws[ks] = wt;
    }
    __syncthreads();
  }

  // 3. update, write the owned entries, mark seeds (a warp's 32 positions are
  //    consecutive, so one ballot gives one word of seed bits)
  if (tid == 0) s_seed[0] = 0u;
  if (tid == 1) s_seed[kChunk / 32 + 1] = 0u;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const int j = c0 + tid + q * kTabThreads;
    const int k = j - base_v;
    bool seed = false;
    if (j < c1) {
      const float v = has_prev ? __fmaf_rn(r, vv[q], s_wv[k]) : vv[q];
      const int d = L - 1 - j;
      float s = 0.f;
      if (d >= 0 && d < N) {
        s = has_prev ? __fmaf_rn(r, sv[q], s_ws[k]) : sv[q];
        sout[d] = s;
      }
      vout[j] = v;
      seed = j >= s_end && j < w_beg && (v > tau || s > tau);
    }
    const uint32_t word = __ballot_sync(0xffffffffu, seed);
    if (lane == 0) s_seed[1 + (tid + q * kTabThreads) / 32] = word;
  }
  __syncthreads();
  if (tid < kHalo) {   // seeds of the halo: positions c0-2, c0-1 and c1, owned by the neighbours
    const int j = tid < 2 ? c0 - 2 + tid : c1;
    const int k = j - base_v;
    bool seed = false;
    if (j >= 0 && j < N && j >= s_end && j < w_beg) {
      const float v = has_prev ? __fmaf_rn(r, __ldg(vin + j), s_wv[k]) : __ldg(vin + j);
      const int d = L - 1 - j;
      float s = 0.f;
      if (d >= 0 && d < N) s = has_prev ? __fmaf_rn(r, __ldg(sin + d), s_ws[k]) : __ldg(sin + d);
      seed = v > tau || s > tau;
    }
    if (seed) {
      const int bit = j - c0 + 32;
      atomicOr(&s_seed[bit >> 5], 1u << (bit & 31));
    }
  }
  // slash entries of negative positions (offset >= L) owned by this chunk
  for (int d = max(c0, L) + tid; d < c1; d += kTabThreads) {
    float s = __ldg(sin + d);
    if (has_prev) {
      const int pos = Lp - 1 - d;                            // >= 0 only if the context shrank
      float w = 0.f;
      if (pos >= 0) {
        bool att = pos < ps_end || pos >= pw_beg;
        if (!att) {
          int lo = 0, hi = scnt;                             // first list entry >= pos
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(sel + mid) < pos) lo = mid + 1; else hi = mid;
          }
          att = lo < scnt && __ldg(sel + lo) == pos;
        }
        if (att) w = attended_weight(logits, pos, lse, one_minus_r);
      }
      s = __fmaf_rn(r, s, w);
    }
    sout[d] = s;
  }
  __syncthreads();

  // 4. expand: position i is a candidate if a seed sits at i-2, i-1, i or i+1
  //    (thread tid takes the consecutive positions jb .., so the compaction
  //    below keeps them ascending)
  const int jb = c0 + kPer * tid;
  uint32_t cbits;
  {
    // bits of positions jb - 2 .. jb + 9 start at bit 8 tid + 30
    const int b0 = kPer * tid + 30;
    const uint64_t w = ((uint64_t)s_seed[(b0 >> 5) + 1] << 32) | s_seed[b0 >> 5];
    const uint32_t win = (uint32_t)(w >> (b0 & 31));          // bit x: position jb - 2 + x
    cbits = (win | (win >> 1) | (win >> 2) | (win >> 3)) & 0xffu;
    // positions outside the middle region or the chunk are no candidates
    const int lo = max(s_end, jb), hi = min(min(w_beg, c1), jb + kPer);
    cbits = hi > lo ? cbits & (((1u << (hi - lo)) - 1u) << (lo - jb)) : 0u;
  }
  const int mine = __popc(cbits);
  // block exclusive scan of the per-thread counts (ascending positions)
  const int x = warp_incl_scan(mine);
  if (lane == 31) s_scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = warp_incl_scan(lane < kTabThreads / 32 ? s_scan[lane] : 0);
    if (lane < kTabThreads / 32) s_scan[lane] = w;
    if (lane == kTabThreads / 32 - 1) s_total = w;
  }
  __syncthreads();
  int pos = (warp > 0 ? s_scan[warp - 1] : 0) + x - mine;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if ((cbits >> q) & 1u) {
      if (pos < cap) stage[pos] = jb + q;
      ++pos;
    }
  }
  if (tid == 0) A.stage_cnt[(size_t)row_id * nch + blockIdx.x] = s_total;
}

// One CTA per (query head, sequence): the chunks' candidates, in chunk
// order, form the ascending candidate list (kcap kept; more is
// SA_ERR_CAPACITY).  The chunk counts are scanned 256 at a time; each warp
// copies whole chunks.
__global__ void __launch_bounds__(256)
tables_compact_kernel(Params p, TableArgs A) {
  pdl_wait();
  pdl_trigger();
  __shared__ int s_off[256];
  __shared__ int s_w[8];
  __shared__ int s_carry;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.mpp * kP;
  const int nch = (N + kChunk - 1) / kChunk;
  const int cap = min(kChunk, p.kcap);
  const int row_id = b * p.Hq + h;
  const int* cnt = A.stage_cnt + (size_t)row_id * nch;
  int* cand = A.cand + (size_t)row_id * p.kcap;
  if (tid == 0) s_carry = 0;
  for (int c0 = 0; c0 < nch; c0 += 256) {
    const int c = c0 + tid;
    const int n = c < nch ? cnt[c] : 0;
    const int x = warp_incl_scan(n);
    if (lane == 31) s_w[warp] = x;
    __syncthreads();
    int before = s_carry + x - n;
    for (int w = 0; w < warp; ++w) before += s_w[w];
    s_off[tid] = before;
    __syncthreads();
    for (int cc = warp; cc < min(256, nch - c0); cc += 8) {
      const int off = s_off[cc];
      const int m = min(cnt[c0 + cc], cap);
      const int* st = A.stage + ((size_t)row_id * nch + c0 + cc) * cap;
      for (int e = lane; e < m && off + e < p.kcap; e += 32) cand[off + e] = st[e];
    }
    __syncthreads();
    if (tid == 255) s_carry = before + n;
    __syncthreads();
  }
  if (tid == 0) {
    const int found = s_carry;
    A.cand_cnt[row_id] = min(found, p.kcap);
    if (found > p.kcap) set_status(A.status, SA_ERR_CAPACITY);
  }
}

size_t tables_stage_bytes(const Params& p) {
  const size_t N = (size_t)p.mpp * kP;
  const size_t nch = (N + kChunk - 1) / kChunk;
  const size_t cap = std::min<size_t>(kChunk, (size_t)std::max(p.kcap, 1));
  return (size_t)p.B * p.Hq * nch * (cap + 1) * sizeof(int);
}

// The staging area at `base` (tables_stage_bytes): candidates, then counts.
void tables_stage_ptrs(const Params& p, void* base, int** stage, int** cnt) {
  const size_t N = (size_t)p.mpp * kP;
  const size_t nch = (N + kChunk - 1) / kChunk;
  const size_t cap = std::min<size_t>(kChunk, (size_t)std::max(p.kcap, 1));
  *stage = static_cast<int*>(base);
  *cnt = *stage + (size_t)p.B * p.Hq * nch * cap;
}

int launch_tables(const Params& p, const TableArgs& A, cudaStream_t stream) {
  const int N = p.mpp * kP;
  const int nch = (N + kChunk - 1) / kChunk;
  cudaError_t e = launch_pdl(tables_kernel, dim3(nch, p.Hq, p.B), dim3(kTabThreads), 0, stream, p, A);
  if (e != cudaSuccess) return SA_ERR_CUDA;
  e = launch_pdl(tables_compact_kernel, dim3(p.Hq, p.B), dim3(256), 0, stream, p, A);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
