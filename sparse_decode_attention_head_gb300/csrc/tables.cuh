// Arguments of the score-table update (tables.cu), shared with the C ABI.
#pragma once

#include "sa_common.cuh"

namespace sa {

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
  const int* frozen;   // [B][Hq] non-zero: the head skipped the previous step (bypass); its tables are copied
  const int* lens;
  int* cand;
  int* cand_cnt;
  int* stage;      // [B * Hq][nchunks][min(kChunk, kcap)] candidates of each chunk
  int* stage_cnt;  // [B * Hq][nchunks]
  int* status;
  float decay;
  float beta;
};

int launch_tables(const Params& p, const TableArgs& A, cudaStream_t stream);
size_t tables_stage_bytes(const Params& p);
void tables_stage_ptrs(const Params& p, void* base, int** stage, int** cnt);

}  // namespace sa
