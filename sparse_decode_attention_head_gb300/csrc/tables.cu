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
// One CTA per (sequence, query head) walks the positions in chunks of
// kChunk: it builds the chunk's weights in shared memory (dense-set entries
// directly, selected tokens from the sorted previous selection list), updates
// and writes both tables (the slash entry tested at position i is offset
// L - 1 - i), marks seeds, expands them, and appends the chunk's candidates
// with a block-wide scan, so the list comes out ascending.  Tables are
// double-buffered (read in, write out) so no CTA reads an entry another has
// already rewritten.
#include "sa_common.cuh"

namespace sa {

constexpr int kTabThreads = 1024;
constexpr int kPer = 4;                        // positions per thread per chunk
constexpr int kChunk = kTabThreads * kPer;     // 4096
constexpr int kHalo = 3;                       // seeds at i-2 .. i+1 expand onto i

struct TableArgs {
  const float* vin;
  const float* sin;
  float* vout;
  float* sout;
  const int* prev_lens;
  const int* prev_sel;
  const int* prev_cnt;
  const float* prev_logits;
  const float* prev_lse;
  const int* lens;
  int* cand;
  int* cand_cnt;
  int* status;
  float decay;
  float beta;
};

// First index in sorted list[0, n) with list[idx] >= x.
__device__ __forceinline__ int lower_bound(const int* list, int n, int x) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(list + mid) < x) lo = mid + 1; else hi = mid;
  }
  return lo;
}

// Fill w[k] = weight of position base + k (k in [0, n)) for the previous step.
__device__ void fill_weights(float* w, int base, int n, const TableArgs& A, const float* logits, int Lp,
                             int ps_end, int pw_beg, const int* sel, int scnt, float lse, float one_minus_r) {
  for (int k = threadIdx.x; k < n; k += blockDim.x) {
    const int pos = base + k;
    float x = 0.f;
    if (pos >= 0 && pos < Lp && (pos < ps_end || pos >= pw_beg))
      x = __fmul_rn(one_minus_r, expf(__ldg(logits + pos) - lse));
    w[k] = x;
  }
  __syncthreads();
  // selected tokens inside the previous middle region (the list is ascending)
  __shared__ int s_range[2];
  if (threadIdx.x == 0) {
    s_range[0] = lower_bound(sel, scnt, max(base, ps_end));
    s_range[1] = lower_bound(sel, scnt, min(base + n, pw_beg));
  }
  __syncthreads();
  for (int e = s_range[0] + threadIdx.x; e < s_range[1]; e += blockDim.x) {
    const int pos = __ldg(sel + e);
    w[pos - base] = __fmul_rn(one_minus_r, expf(__ldg(logits + pos) - lse));
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kTabThreads)
tables_kernel(Params p, TableArgs A) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_wv[kChunk + kHalo];       // weights feeding the vertical entries (positions c0-2 ..)
  __shared__ float s_ws[kChunk + kHalo];       // weights feeding the slash entries tested there
  __shared__ unsigned char s_seed[kChunk + kHalo];
  __shared__ int s_scan[32];
  __shared__ int s_total;

  const int h = blockIdx.x, b = blockIdx.y;
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
  const bool has_prev = A.prev_logits != nullptr;
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
  int* cand = A.cand + ((size_t)b * p.Hq + h) * p.kcap;
  int found = 0;

  for (int c0 = 0; c0 < N; c0 += kChunk) {
    const int c1 = min(N, c0 + kChunk);
    const int n = c1 - c0 + kHalo;                           // positions c0-2 .. c1
    if (has_prev) {
      fill_weights(s_wv, c0 - 2, n, A, logits, Lp, ps_end, pw_beg, sel, scnt, lse, one_minus_r);
      fill_weights(s_ws, c0 - 2 - delta, n, A, logits, Lp, ps_end, pw_beg, sel, scnt, lse, one_minus_r);
    }
    // update, write owned entries, mark seeds
    for (int k = tid; k < n; k += blockDim.x) {
      const int j = c0 - 2 + k;                              // position
      bool seed = false;
      if (j >= 0 && j < N) {
        const float v = has_prev ? __fmaf_rn(r, __ldg(vin + j), s_wv[k]) : __ldg(vin + j);
        const int d = L - 1 - j;                             // slash offset of position j
        float s = 0.f;
        if (d >= 0 && d < N) s = has_prev ? __fmaf_rn(r, __ldg(sin + d), s_ws[k]) : __ldg(sin + d);
        if (j >= c0 && j < c1) {                             // owned: write
          vout[j] = v;
          if (d >= 0 && d < N) sout[d] = s;
        }
        seed = j >= s_end && j < w_beg && (v > tau || s > tau);
      }
      s_seed[k] = seed;
    }
    // slash entries of negative positions (offset >= L) owned by this chunk
    for (int d = max(c0, L) + tid; d < c1; d += blockDim.x) {
      float s = __ldg(sin + d);
      if (has_prev) {
        const int pos = Lp - 1 - d;                          // >= 0 only if the context shrank
        float w = 0.f;
        if (pos >= 0) {
          bool att = pos < ps_end || pos >= pw_beg;
          if (!att) {
            const int e = lower_bound(sel, scnt, pos);
            att = e < scnt && __ldg(sel + e) == pos;
          }
          if (att) w = __fmul_rn(one_minus_r, expf(__ldg(logits + pos) - lse));
        }
        s = __fmaf_rn(r, s, w);
      }
      sout[d] = s;
    }
    __syncthreads();
    // expand: position i is a candidate if a seed sits at i-2, i-1, i or i+1
    int mine = 0;
    bool is_c[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int i = c0 + tid * kPer + q;
      const int k = i - (c0 - 2);
      bool cnd = false;
      if (i < c1 && i >= s_end && i < w_beg)
        cnd = s_seed[k - 2] | s_seed[k - 1] | s_seed[k] | s_seed[k + 1];
      is_c[q] = cnd;
      mine += cnd;
    }
    // block exclusive scan of the per-thread counts (ascending positions)
    int x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s_scan[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = s_scan[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      s_scan[lane] = w;
      if (lane == 31) s_total = w;
    }
    __syncthreads();
    int pos = found + (warp > 0 ? s_scan[warp - 1] : 0) + x - mine;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      if (is_c[q]) {
        if (pos < p.kcap) cand[pos] = c0 + tid * kPer + q;
        ++pos;
      }
    }
    found += s_total;
    __syncthreads();
  }
  if (tid == 0) {
    A.cand_cnt[(size_t)b * p.Hq + h] = min(found, p.kcap);
    if (found > p.kcap) set_status(A.status, SA_ERR_CAPACITY);
  }
}

int launch_tables(const Params& p, const TableArgs& A, cudaStream_t stream) {
  dim3 grid(p.Hq, p.B);
  const cudaError_t e = launch_pdl(tables_kernel, grid, dim3(kTabThreads), 0, stream, p, A);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
