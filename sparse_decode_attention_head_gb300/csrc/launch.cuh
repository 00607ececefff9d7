// Host entry points of the kernels (one definition each, in the .cu file
// named beside it), shared by the C ABI (sa_api.cu) and the allocation-free
// decode (noalloc.cu), and the host helpers of the C ABI that noalloc.cu uses.
#pragma once

#include <cuda.h>

#include "sa_common.cuh"
#include "sparsity.cuh"
#include "tables.cuh"

namespace sa {
// summarize.cu, select.cu, merge.cu, decode.cu, step.cu, tokens.cu, bypass.cu
int launch_summarize(const Params& p, const void* k_pool, const int* page_table, const int* seq_lens,
                     int block_begin, int block_end, void* summ, int* status, cudaStream_t stream);
int launch_score(const Params& p, const void* q, const void* summ, const int* seq_lens, float* scores,
                 int always, int num_sms, cudaStream_t stream, const EstArgs* est);
int launch_topk(const Params& p, const float* scores, const int* seq_lens, int* sel_idx, int* sel_cnt,
                cudaStream_t stream);
size_t topk_smem_bytes(const Params& p);
int launch_build_tiles(const Params& p, const int* seq_lens, const int* page_table, const int* sel_idx,
                       const int* sel_cnt, int gran, void* tiles, int* ntiles, int* status, int* ticket,
                       cudaStream_t stream);
int launch_decode(const Params& p, const void* q, const int* page_table, const void* tiles, const int* ntiles,
                  float* partials, int* ticket, float* out, float* lse, float* logits, int* status,
                  const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms, cudaStream_t stream);
size_t decode_smem_bytes(const Params& p);
size_t decode_partials_bytes(const Params& p);
size_t tiles_bytes(const Params& p);
size_t ntiles_bytes(const Params& p);
int launch_lse_merge(int n_rows, int D, const float* o_a, const float* lse_a, const float* o_b,
                     const float* lse_b, float* o, float* lse, cudaStream_t stream);
int launch_build_step(const Params& p, const int* seq_lens, const int* page_table, void* k_pool, void* v_pool,
                      const void* k_new, const void* v_new, float* stats, void* summ, const int* sel_idx, int* sel_cnt,
                      void* tiles, int* ntiles, int* status, int* ticket, cudaStream_t stream);
int launch_append_kv(const Params& p, const int* seq_lens, const int* page_table, const void* k_new, const void* v_new,
                     void* k_pool, void* v_pool, int* status, cudaStream_t stream);
int launch_token_topk(const Params& p, const void* q, const void* k_pool, const int* page_table, const int* seq_lens,
                      const int* cand_idx, const int* cand_cnt, int* sel_idx, int* sel_cnt, float* scores_out,
                      int* status, cudaStream_t stream);
int launch_select_build(const Params& p, const float* scores, const int* seq_lens, const int* page_table,
                        void* k_pool, void* v_pool, const void* k_new, const void* v_new, float* stats, void* summ,
                        int* sel_idx, int* sel_cnt, void* tiles, int* ntiles, int* status, int* ticket,
                        cudaStream_t stream);
int launch_kv_stats(const Params& p, const void* k_pool, const void* v_pool, const int* page_table,
                    const int* seq_lens, float* stats, int* status, cudaStream_t stream);
int launch_sparsity(const Params& p, const void* q, const int* seq_lens, const EstArgs& E, cudaStream_t stream);
}  // namespace sa

namespace sa_host {
// sa_api.cu
int make_params(const sa_problem* pr, sa::Params* p);
int make_kv_map(CUtensorMap* m, const void* pool, const sa::Params& p);
int num_sms_current();
}  // namespace sa_host
