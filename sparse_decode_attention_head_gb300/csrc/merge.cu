// Step a6 as a standalone call: the exact log-sum-exp fusion of two partial
// attentions over disjoint key sets (HGCA review, "What carries the
// argument"), stabilised by the larger lse (minor comment on Sec. 3.3).
// One warp per row; elementwise and HBM-bound.
#include "sa_common.cuh"

namespace sa {

__global__ void lse_merge_kernel(int n_rows, int D, const float* o_a, const float* lse_a, const float* o_b,
                                 const float* lse_b, float* o, float* lse) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < n_rows; r += warps) {
    const float la = lse_a[r], lb = lse_b[r];
    const float m = fmaxf(la, lb);
    float wa = 0.f, wb = 0.f;
    if (m != -INFINITY) {
      wa = la == -INFINITY ? 0.f : expf(la - m);
      wb = lb == -INFINITY ? 0.f : expf(lb - m);
    }
    const float den = wa + wb;
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const size_t base = (size_t)r * D;
    for (int d = lane; d < D; d += 32) {
      const float xa = wa != 0.f ? o_a[base + d] : 0.f;
      const float xb = wb != 0.f ? o_b[base + d] : 0.f;
      o[base + d] = (wa * xa + wb * xb) * inv;
    }
    __syncwarp();
    if (lane == 0) lse[r] = den > 0.f ? m + logf(den) : -INFINITY;
  }
}

int launch_lse_merge(int n_rows, int D, const float* o_a, const float* lse_a, const float* o_b,
                     const float* lse_b, float* o, float* lse, cudaStream_t stream) {
  if (n_rows == 0) return SA_OK;
  const int threads = 256;
  long long blocks = ((long long)n_rows * 32 + threads - 1) / threads;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  const cudaError_t e =
      launch_pdl(lse_merge_kernel, dim3((int)blocks), dim3(threads), 0, stream, n_rows, D, o_a, lse_a, o_b, lse_b, o, lse);
  return e == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // namespace sa
