// Internal declarations shared by the host planner, the entry points and the
// kernels.  Not part of the public C ABI (include/pkv.h is).
#pragma once

#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int32_t kPlanMagic = 0x31564b50;  // "PKV1"
constexpr int kBlockSize = 16;
constexpr int kRowsPerTile = 16;    // query rows (token x head-in-group) per decode tile
constexpr int kPrefillRows = 128;   // query rows per tensor-core tile

// Plan buffer: [PlanHeader][DecodeTile x n][MergeGroup x m][PrefillTile x k]
struct PlanHeader {
  int32_t magic;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t total_q;
  int32_t num_decode_tiles;
  int32_t num_merge_groups;
  int32_t num_prefill_tiles;
  int32_t num_partials;
  int32_t split_blocks;
  int32_t max_blocks_needed;
  int32_t reserved[4];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

// One split-KV work item.  Runs once per KV head (grid.y).  Covers query
// tokens qi0 .. qi0+n_q-1 of sequence `seq` (all heads of the GQA group, so
// n_q * group <= 16 rows) against logical KV blocks [kb_begin, kb_end).
struct DecodeTile {
  int32_t seq;
  int32_t qi0;       // first query token, relative to the sequence's chunk
  int32_t n_q;       // query tokens in the row group
  int32_t kb_begin;  // first logical KV block
  int32_t kb_end;    // one past the last logical KV block
  int32_t part;      // partial slot, or -1: the only split, write `out` directly
  int32_t last;      // 1 if this split ends at the row group's last needed block
  int32_t pad;
};
static_assert(sizeof(DecodeTile) == 32, "decode tile is 32 bytes");

// Row group whose keys were split over `nsplit` tiles with consecutive
// partial slots part0 .. part0+nsplit-1.
struct MergeGroup {
  int32_t seq;
  int32_t qi0;
  int32_t n_q;
  int32_t part0;
  int32_t nsplit;
  int32_t pad[3];
};
static_assert(sizeof(MergeGroup) == 32, "merge group is 32 bytes");

// Tensor-core work item: 128 query tokens of one sequence x one query head.
struct PrefillTile {
  int32_t seq;
  int32_t qi0;
  int32_t hq;
  int32_t n_q;
};
static_assert(sizeof(PrefillTile) == 16, "prefill tile is 16 bytes");

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Byte offsets inside the plan buffer, from the counts alone.
inline int64_t plan_decode_off() { return (int64_t)sizeof(PlanHeader); }
inline int64_t plan_merge_off(int32_t n_decode) {
  return plan_decode_off() + (int64_t)n_decode * (int64_t)sizeof(DecodeTile);
}
inline int64_t plan_prefill_off(int32_t n_decode, int32_t n_merge) {
  return plan_merge_off(n_decode) + (int64_t)n_merge * (int64_t)sizeof(MergeGroup);
}

// Workspace: partial O [num_partials][Hkv][16][D] fp32, then (m, l) pairs
// [num_partials][Hkv][16] float2.
inline int64_t ws_part_o_bytes(int32_t parts, int32_t hkv, int32_t d) {
  return align_up((int64_t)parts * hkv * kRowsPerTile * d * 4, 256);
}
inline int64_t ws_part_ml_bytes(int32_t parts, int32_t hkv) {
  return align_up((int64_t)parts * hkv * kRowsPerTile * 8, 256);
}

// Kernel launchers (defined in the .cu files).  Return a cudaError_t value.
int launch_append(const void *k, const void *v, const int32_t *slot_mapping, int32_t num_tokens,
                  void *kv_pool, const pkv_pool_desc &desc, int32_t *dev_status,
                  pkv_stream stream);

struct AttnArgs {
  const void *q;
  void *out;
  const int32_t *cu_q_lens;
  const int32_t *context_lens;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  const void *kv_pool;
  pkv_pool_desc desc;
  int32_t num_q_heads;
  int32_t num_seqs;
  float scale;
  const DecodeTile *decode_tiles;
  int32_t num_decode_tiles;
  const MergeGroup *merge_groups;
  int32_t num_merge_groups;
  const PrefillTile *prefill_tiles;
  int32_t num_prefill_tiles;
  float *part_o;
  float *part_ml;
  int32_t *dev_status;
  pkv_stream stream;
};

int launch_decode(const AttnArgs &a, int *launches);
int launch_merge(const AttnArgs &a, int *launches);

void count_launches(int n);

// Profiling hook (pkv_set_profile_events): events recorded around launches of
// one kernel id on the launching stream; per host thread.
void profile_begin(int which, pkv_stream stream);
void profile_end(int which, pkv_stream stream);

}  // namespace pkv
