// Host step metadata: validates one packed step's lengths and cuts it into
// work tiles for the attention kernels.
//
// The vllm-metal kernel ("Replacing attention, reusing the rest") has every
// threadgroup binary-search cu_seqlens to find the request owning its query
// token.  Here the scheduler's host copies of cu_q_lens / context_lens are
// turned into an explicit tile list once per step instead, so every CTA reads
// its (sequence, query rows, key range) directly.
//
// Tiling:
//  * Query rows of a sequence are grouped GQA-first: a row group holds n_q
//    consecutive query tokens x all `group` query heads of one KV head, with
//    n_q * group <= 16 (one m16 MMA tile), so each KV block loaded serves every
//    query head that reads it.
//  * A row group's keys [0, last visible key] are cut into splits of about
//    `split_blocks` 16-token blocks.  split_blocks is chosen from the total
//    work so that the decode grid is ~4 CTAs per SM (2 resident x 2 waves);
//    row groups with several splits get partial-result slots and a merge group.
//  * Tiles are ordered longest first so the hardware block scheduler deals the
//    long ones out before the short ones (longest-processing-time order).
#include <algorithm>
#include <cstring>
#include <vector>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kMinSplitBlocks = 16;
constexpr int kMaxSplitBlocks = 1024;
constexpr int kCtasPerSmTarget = 4;

pkv_status check_desc(const pkv_pool_desc *desc, int32_t num_q_heads) {
  if (!desc) return PKV_ERR_NULL;
  if (desc->block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (desc->num_kv_heads < 1 || desc->num_blocks < 0) return PKV_ERR_SHAPE;
  if (num_q_heads < 1 || num_q_heads % desc->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (num_q_heads / desc->num_kv_heads > kRowsPerTile) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

struct RowGroup {
  int32_t seq, qi0, n_q, nb;
};

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_plan_step(const int32_t *cu_q_lens, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    const pkv_pool_desc *desc, int32_t num_sms, void *plan,
                                    int64_t plan_capacity, pkv_plan_info *info) {
  if (!info) return PKV_ERR_NULL;
  pkv_status st = check_desc(desc, num_q_heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0) return PKV_ERR_SHAPE;
  if (num_seqs > 0 && (!cu_q_lens || !context_lens)) return PKV_ERR_NULL;
  if (num_sms <= 0) num_sms = 152;

  const int32_t hkv = desc->num_kv_heads;
  const int32_t group = num_q_heads / hkv;
  const int32_t nq_tile = std::max(1, kRowsPerTile / group);

  // ---- validate and build row groups
  if (num_seqs > 0 && cu_q_lens[0] != 0) return PKV_ERR_SHAPE;
  std::vector<RowGroup> groups;
  int64_t kv_tokens = 0, total_blocks = 0;
  int32_t max_nb = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t qs64 = (int64_t)cu_q_lens[s + 1] - (int64_t)cu_q_lens[s];
    if (qs64 < 0) return PKV_ERR_SHAPE;
    int32_t qs = (int32_t)qs64, ctx = context_lens[s];
    if (ctx < 0 || qs > ctx) return PKV_ERR_RANGE;
    if (qs == 0) continue;
    kv_tokens += ctx;
    max_nb = std::max(max_nb, (ctx + kBlockSize - 1) / kBlockSize);
    for (int32_t qi0 = 0; qi0 < qs; qi0 += nq_tile) {
      int32_t n_q = std::min(nq_tile, qs - qi0);
      int32_t last_key = ctx - qs + qi0 + n_q - 1;
      int32_t nb = last_key / kBlockSize + 1;
      groups.push_back({s, qi0, n_q, nb});
      total_blocks += nb;
    }
  }

  // ---- split size from the total work
  int64_t units = total_blocks * hkv;
  int64_t target = (int64_t)num_sms * kCtasPerSmTarget;
  int64_t split = (units + target - 1) / std::max<int64_t>(target, 1);
  split = std::min<int64_t>(std::max<int64_t>(split, kMinSplitBlocks), kMaxSplitBlocks);

  std::vector<DecodeTile> tiles;
  std::vector<MergeGroup> merges;
  int32_t parts = 0;
  for (const RowGroup &g : groups) {
    int32_t nsplit = (int32_t)((g.nb + split - 1) / split);
    int32_t per = (g.nb + nsplit - 1) / nsplit;
    nsplit = (g.nb + per - 1) / per;
    int32_t part0 = nsplit > 1 ? parts : -1;
    for (int32_t j = 0; j < nsplit; ++j) {
      DecodeTile t;
      t.seq = g.seq;
      t.qi0 = g.qi0;
      t.n_q = g.n_q;
      t.kb_begin = j * per;
      t.kb_end = std::min(g.nb, (j + 1) * per);
      t.part = nsplit > 1 ? part0 + j : -1;
      t.last = (j == nsplit - 1) ? 1 : 0;
      t.pad = 0;
      tiles.push_back(t);
    }
    if (nsplit > 1) {
      MergeGroup m;
      std::memset(&m, 0, sizeof m);
      m.seq = g.seq;
      m.qi0 = g.qi0;
      m.n_q = g.n_q;
      m.part0 = part0;
      m.nsplit = nsplit;
      merges.push_back(m);
      parts += nsplit;
    }
  }
  std::stable_sort(tiles.begin(), tiles.end(), [](const DecodeTile &a, const DecodeTile &b) {
    return (a.kb_end - a.kb_begin) > (b.kb_end - b.kb_begin);
  });

  // ---- sizes
  std::memset(info, 0, sizeof *info);
  info->num_seqs = num_seqs;
  info->num_q_heads = num_q_heads;
  info->num_kv_heads = hkv;
  info->head_dim = desc->head_dim;
  info->total_q = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
  info->num_decode_tiles = (int32_t)tiles.size();
  info->num_merge_groups = (int32_t)merges.size();
  info->num_partials = parts;
  info->num_prefill_tiles = 0;
  info->num_kernels = (tiles.empty() ? 0 : 1) + (merges.empty() ? 0 : 1);
  info->split_blocks = (int32_t)split;
  info->max_blocks_needed = max_nb;
  info->kv_tokens = kv_tokens;
  info->plan_bytes = plan_prefill_off(info->num_decode_tiles, info->num_merge_groups);
  info->workspace_bytes =
      parts > 0 ? ws_part_o_bytes(parts, hkv, desc->head_dim) + ws_part_ml_bytes(parts, hkv) : 0;

  if (!plan) return PKV_OK;
  if (plan_capacity < info->plan_bytes) return PKV_ERR_WORKSPACE;
  PlanHeader h;
  std::memset(&h, 0, sizeof h);
  h.magic = kPlanMagic;
  h.num_seqs = num_seqs;
  h.num_q_heads = num_q_heads;
  h.num_kv_heads = hkv;
  h.head_dim = desc->head_dim;
  h.total_q = info->total_q;
  h.num_decode_tiles = info->num_decode_tiles;
  h.num_merge_groups = info->num_merge_groups;
  h.num_prefill_tiles = 0;
  h.num_partials = parts;
  h.split_blocks = (int32_t)split;
  h.max_blocks_needed = max_nb;
  char *p = static_cast<char *>(plan);
  std::memcpy(p, &h, sizeof h);
  if (!tiles.empty())
    std::memcpy(p + plan_decode_off(), tiles.data(), tiles.size() * sizeof(DecodeTile));
  if (!merges.empty())
    std::memcpy(p + plan_merge_off(info->num_decode_tiles), merges.data(),
                merges.size() * sizeof(MergeGroup));
  return PKV_OK;
}
