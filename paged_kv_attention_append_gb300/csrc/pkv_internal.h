// Internal declarations shared by the host planner, the entry points and the
// kernels.  Not part of the public C ABI (include/pkv.h is).
#pragma once

#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int32_t kPlanMagic = 0x33564b50;  // "PKV3"
constexpr int kBlockSize = 16;
constexpr int kRowsPerTile = 16;    // query rows (token x head-in-group) per decode row group
constexpr int kPrefillRows = 128;   // query tokens per tensor-core tile
constexpr int kDecodeWarpsPerCta = 4;

// Plan buffer layout (all offsets are functions of the counts):
//   [PlanHeader 64 B]
//   [warp_begin: int32 x (num_decode_warps + 1), padded to 32 B]
//   [warp_head: WarpHead x num_decode_warps] (each warp's first piece and, when
//    the planner was given the host block tables, its first blocks' physical
//    ids: a warp reads its range and head with two independent loads and can
//    start its first copies without waiting for a block-table read)
//   [Piece x num_decode_pieces][MergeGroup x num_merge_groups]
//   [SharedItem x num_shared_items]  (pair k's first item at index k)
//   [prefill_begin: int32 x (num_prefill_ctas + 1), padded to 32 B; absent when 0 CTAs]
//   [PrefillTile x num_prefill_tiles, grouped by CTA]
//   [GatherRow x num_gather_rows] (the query tokens of gathered sub-tiles)
struct PlanHeader {
  int32_t magic;
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t total_q;
  int32_t num_decode_warps;
  int32_t num_decode_pieces;
  int32_t num_merge_groups;
  int32_t num_partials;
  int32_t num_prefill_tiles;
  int32_t max_blocks_needed;
  int32_t reserved[4];
};
static_assert(sizeof(PlanHeader) == 64, "plan header is 64 bytes");

// A contiguous key range of one (row group, KV head) segment, processed by one
// warp of the split-KV kernel.  A row group is n_q consecutive query tokens of
// sequence `seq` x all query heads of KV head h (n_q * group <= 16 rows).
struct Piece {
  int32_t seq;
  int32_t qi0;       // first query token of the row group, relative to the sequence's chunk
  int32_t n_q;       // query tokens in the row group
  int32_t h;         // KV head
  int32_t kb_begin;  // first logical KV block of the piece
  int32_t kb_end;    // one past the last logical KV block of the piece
  int32_t part;      // partial slot, or -1 when the piece is the whole segment (writes out)
  int32_t q_row0;    // packed query index of token qi0 (cu_q_lens[seq] + qi0)
};
static_assert(sizeof(Piece) == 32, "piece is 32 bytes");

// Per-warp head of the split-KV work: a copy of the warp's first piece, and
// the physical block ids of that piece's first kHeadBlocks blocks (-1 where not
// known at planning time or past the piece).
constexpr int kHeadBlocks = 3;
struct WarpHead {
  Piece first;
  int32_t blk[4];
};
static_assert(sizeof(WarpHead) == 48, "warp head is 48 bytes");

// Shared-block work for one pair of split-KV warps (a CTA has
// kSharedItemsPerCta pairs; pair k of the shared CTAs starts with item k and
// runs the items chained from it through `next`, which is -1 after the last
// and otherwise a later index): row groups that read the same blocks -- of one
// verify window wider than 16 rows, or of sequences whose block tables start
// with the same physical blocks -- read them once, each of the pair's warps
// attending one row group to every loaded block.  Blocks kb_begin .. kb_end-1 of
// sequence seq0's table, KV head h; warp w < n_rg of the pair takes row group
// rg[w] and writes its partial to rg[w].part (or its result directly when part
// < 0).  n_rg == 0: an empty item (its pair idles).
struct SharedRowGroup {
  int32_t seq;
  int32_t qi0;
  int32_t n_q;
  int32_t part;
  int32_t q_row0;  // packed query index of token qi0
  int32_t pad[3];
};
constexpr int kSharedRowGroups = 2;   // row groups (warps) per shared item
constexpr int kSharedItemsPerCta = kDecodeWarpsPerCta / kSharedRowGroups;
struct SharedItem {
  int32_t seq0;
  int32_t h;
  int32_t kb_begin;
  int32_t kb_end;
  int32_t n_rg;
  int32_t next;  // the pair's next item, or -1
  int32_t pad[2];
  SharedRowGroup rg[kSharedRowGroups];
};
static_assert(sizeof(SharedItem) == 32 + 32 * kSharedRowGroups, "shared item layout");

// A set of nsplit partial results (slots part0 .. part0+nsplit-1) to combine.
// kind 0: a decode segment -- rows are n_q tokens x the group's heads of KV
//         head h, partial slots of kRowsPerTile rows;
// kind 1: a prefill sub-tile cut along its keys -- rows are the n_q tokens of
//         query head h (here a query head), partial slots of kPrefillRows rows.
struct MergeGroup {
  int32_t seq;
  int32_t qi0;
  int32_t n_q;
  int32_t h;
  int32_t part0;
  int32_t nsplit;
  int32_t kind;
  int32_t q_row0;  // packed query index of token qi0 (cu_q_lens[seq] + qi0)
};
static_assert(sizeof(MergeGroup) == 32, "merge group is 32 bytes");

// Tensor-core work item: up to two query sub-tiles whose query heads share KV
// head h, so every K/V tile loaded serves both; keys are read through sequence
// seq's block table.  The item covers key tiles kt0 .. kt1-1 (128 keys each).
// n_q[1] == 0 means a single sub-tile.  Sub-tile x is either
//  * contiguous (gather[x] < 0): query tokens qi0[x] .. qi0[x]+n_q[x]-1 (n_q <=
//    128) of sequence seq, query head hq[x], causal; sub-tile 0 sees at least as
//    many keys as sub-tile 1.  A sub-tile whose keys the item covers only in
//    part writes its unnormalised result to prefill partial slot part[x] (else
//    part[x] = -1 and it writes out directly); or
//  * gathered (gather[x] >= 0): rows (token t, head g) = row t * G + g for the
//    n_q[x] tokens GatherRow[gather[x] ..] (n_q * G <= 128), all G query heads
//    of KV head h, tokens of any sequences whose tables hold the same physical
//    blocks over the item's keys, every key visible to every row (no mask).
//    Row (t, g) writes its unnormalised result to decode partial slot
//    GatherRow.part0 + part[x], row GatherRow.row0 + g.  When bit x of `runs`
//    is set the tokens are consecutive packed indices from qi0[x] (loaded as
//    one box of 128 / G tokens).
struct PrefillTile {
  int32_t seq;
  int32_t h;
  int32_t hq[2];
  int32_t qi0[2];
  int32_t n_q[2];
  int32_t kt0;
  int32_t kt1;
  int32_t part[2];
  int32_t gather[2];
  int32_t runs;
  int32_t pad;
};
static_assert(sizeof(PrefillTile) == 64, "prefill tile is 64 bytes");

// One query token of a gathered sub-tile: its packed index, the decode partial
// slot its row group's first key chunk writes, and the row of its first head in
// that slot.
struct GatherRow {
  int32_t q_tok;
  int32_t part0;
  int32_t row0;
  int32_t pad;
};
static_assert(sizeof(GatherRow) == 16, "gather row is 16 bytes");

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

struct PlanOffsets {
  int64_t warp_begin, warp_head, pieces, merges, shared, prefill_begin, prefill, gather, total;
};
inline PlanOffsets plan_offsets(int32_t n_warps, int32_t n_pieces, int32_t n_merge,
                                int32_t n_shared, int32_t n_prefill, int32_t n_prefill_ctas,
                                int32_t n_gather) {
  PlanOffsets o;
  o.warp_begin = (int64_t)sizeof(PlanHeader);
  o.warp_head = o.warp_begin + align_up(4ll * (n_warps + 1), 32);
  o.pieces = o.warp_head + (int64_t)n_warps * (int64_t)sizeof(WarpHead);
  o.merges = o.pieces + (int64_t)n_pieces * (int64_t)sizeof(Piece);
  o.shared = o.merges + (int64_t)n_merge * (int64_t)sizeof(MergeGroup);
  o.prefill_begin = o.shared + (int64_t)n_shared * (int64_t)sizeof(SharedItem);
  o.prefill = o.prefill_begin + (n_prefill_ctas > 0 ? align_up(4ll * (n_prefill_ctas + 1), 32) : 0);
  o.gather = o.prefill + (int64_t)n_prefill * (int64_t)sizeof(PrefillTile);
  o.total = o.gather + (int64_t)n_gather * (int64_t)sizeof(GatherRow);
  return o;
}

// Workspace: decode partial O [num_partials][16][D] fp32, then (m, l) pairs
// [num_partials][16] float2 (only the row group's rows are written); then
// prefill partial O [num_prefill_partials][128][D] fp32 and (m, l)
// [num_prefill_partials][128] float2.
inline int64_t ws_part_o_bytes(int32_t parts, int32_t d) {
  return align_up((int64_t)parts * kRowsPerTile * d * 4, 256);
}
inline int64_t ws_part_ml_bytes(int32_t parts) {
  return align_up((int64_t)parts * kRowsPerTile * 8, 256);
}
inline int64_t ws_ppart_o_bytes(int32_t pparts, int32_t d) {
  return align_up((int64_t)pparts * kPrefillRows * d * 4, 256);
}
inline int64_t ws_ppart_ml_bytes(int32_t pparts) {
  return align_up((int64_t)pparts * kPrefillRows * 8, 256);
}
inline int64_t ws_total_bytes(int32_t parts, int32_t pparts, int32_t d) {
  return ws_part_o_bytes(parts, d) + ws_part_ml_bytes(parts) + ws_ppart_o_bytes(pparts, d) +
         ws_ppart_ml_bytes(pparts);
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
  int64_t total_q;
  float scale;
  const int32_t *warp_begin;
  const WarpHead *warp_head;
  int32_t num_decode_warps;
  const SharedItem *shared_items;
  int32_t num_shared_ctas;
  int32_t num_shared_items;   // SharedItem entries (the CTAs' pairs' chains)
  const Piece *pieces;
  const MergeGroup *merge_groups;
  int32_t num_merge_groups;
  const int32_t *prefill_begin;
  const PrefillTile *prefill_tiles;
  const GatherRow *gather_rows;
  int32_t num_gather_rows;
  int32_t num_partials;       // decode partial slots (gathered sub-tiles write into them)
  int32_t num_prefill_tiles;
  int32_t num_prefill_ctas;
  float *part_o;
  float *part_ml;
  float *ppart_o;
  float *ppart_ml;
  int32_t num_decode_merges;  // merge_groups[0 .. num_decode_merges) are kind 0
  int32_t merge_rows;         // rows of the largest decode merge group
  int32_t lookahead;          // further decode steps the plan covers (chained decode)
  int32_t *dev_status;
  pkv_stream stream;
};

int launch_state_checkpoint(const void *src, const int32_t *dst_slots, int32_t num_rows,
                            void *pool, int64_t num_slots, int64_t row_bytes, int32_t *dev_status,
                            pkv_stream stream);

int launch_decode_advance(int32_t *context_lens, int32_t *slot_mapping, const int32_t *cu_q_lens,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          int32_t num_seqs, int32_t num_blocks, int32_t *dev_status,
                          pkv_stream stream);

int launch_decode(const AttnArgs &a, int *launches);
int launch_merge(const AttnArgs &a, int *launches);
int launch_prefill(const AttnArgs &a, int *launches);

// 4-D TMA view of the pool whose box is one paged block of one head, landing
// as [8-row group][64-column half][8 rows][128 B], 128-byte swizzled; `map`
// points to a CUtensorMap.
int make_pool_map(void *map, const void *pool, const pkv_pool_desc &desc);

void count_launches(int n);

// Streaming multiprocessors of the calling thread's current device (cached per
// device); 0 when no device can be queried.
int device_sm_count();

// Profiling hook (pkv_set_profile_events): events recorded around launches of
// one kernel id on the launching stream; per host thread.
void profile_begin(int which, pkv_stream stream);
void profile_end(int which, pkv_stream stream);
// True when any profiling event is set on this host thread; kernels are then
// launched without programmatic stream serialisation so events bracket them.
bool profiling_active();

}  // namespace pkv
