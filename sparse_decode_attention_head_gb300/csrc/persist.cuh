// The persistent decode step (persist.cu): arguments, the global hand-off
// state it keeps in the workspace, and its host entry points.
#pragma once

#include <cuda.h>

#include "sa_common.cuh"
#include "tiles.cuh"

namespace sa {

constexpr int kPMaxC = 32;              // tiles per chunk at most (a chunk is staged whole in shared memory)
constexpr int kPMaxChunksUnit = 1024;   // chunks per (sequence, KV head) at most
constexpr int kPMaxUnits = 1024;        // (sequence, KV head) units per launch at most

// Global hand-off state (ints in the workspace; zero between launches):
// tickets and counts, then per unit: blocks scored, heads selected, chunks
// combined, and its first queue position and chunk count + 1 (0: not built).
constexpr int kGsScoreTicket = 0, kGsSelTicket = 1, kGsQTail = 2, kGsQHead = 3, kGsUnitsBuilt = 4, kGsExit = 5,
              kGsMergeTicket = 6;
constexpr int kGsHead = 8;
constexpr int kGsPerUnit = 5;

// One chunk of a unit's tile list in the global queue; `flag` is set last.
struct PQEntry {
  int unit, t0, nt, nch, pos0, kin, flag, pad;
};

struct PArgs {
  const __nv_bfloat16* q;
  const __nv_bfloat16* summ_r;   // summaries read by the scores
  __nv_bfloat16* summ_w;         // step: the tail block rewritten here (NULL: no refresh)
  const __nv_bfloat16* k_pool;   // read by the tail refresh
  const int* page_table;
  const int* seq_lens;
  int* sel_idx;                  // step: written; given selections: read
  int* sel_cnt;
  float* scores;                 // [B][Hq][slots]
  Tile* tiles;                   // [B * Hk][max_pages_per_seq]
  float* partials;               // [qcap][partial_stride(G)]
  int* gs;                       // hand-off state (persist_gs_bytes)
  PQEntry* dq;                   // [qcap]
  float* out;
  float* lse;
  int* status;
  int qcap;
  int C;                         // tiles per chunk
  int given;                     // 1: selections given (no scores, no top-k)
  int nslots;                    // slots per consumer warp
};

int persist_chunk_tiles(const Params& p);
size_t persist_qcap(const Params& p);
size_t persist_gs_bytes(const Params& p);
size_t persist_partials_bytes(const Params& p);
bool persist_supported(const Params& p, bool step);
int launch_persist(const Params& p, const PArgs& A, const CUtensorMap& tmK, const CUtensorMap& tmV, int num_sms,
                   cudaStream_t stream);

}  // namespace sa
