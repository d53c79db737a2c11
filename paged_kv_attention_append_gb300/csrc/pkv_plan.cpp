// Host step metadata: validates one packed step's lengths and cuts it into
// work for the attention kernels.
//
// The vllm-metal kernel ("Replacing attention, reusing the rest") has every
// threadgroup binary-search cu_seqlens to find the request owning its query
// token.  Here the scheduler's host copies of cu_q_lens / context_lens are
// turned into explicit work lists once per step instead.
//
// Decode-class rows (split-KV kernel):
//  * Query rows of a sequence are grouped GQA-first: a row group holds n_q
//    consecutive query tokens x all `group` query heads of one KV head, with
//    n_q * group <= 16 (one m16 MMA tile), so each KV block loaded serves every
//    query head that reads it.  A segment is (row group, KV head) with the
//    blocks [0, last visible key / 16].
//  * All segments' blocks are laid end to end and cut into num_decode_warps
//    contiguous ranges of equal cost (blocks plus a fixed charge per segment
//    start), one per warp (8 warps per SM, one wave).  A range
//    intersects one or more segments; each intersection is a piece.  A segment
//    cut into several pieces gets one partial slot per piece and a merge group.
//    Equal ranges leave no tail wave and no long/short CTA imbalance.
//
// Shared prefixes (when the planner has the host block tables): decode-class
// sequences whose tables start with the same physical blocks read those blocks
// once per work unit rather than once per row group.  When at least 64 query
// rows per KV head share a prefix of whole 128-key tiles, the prefix goes to the
// tensor-core kernel as gathered sub-tiles: 128 rows (token x query head) taken
// from all those sequences attend one key tile per MMA, each row writing a
// partial result that the merge combines with its own suffix.  Smaller groups
// use split-KV CTAs whose warp pairs stream the prefix once for two row groups
// (as the two row groups of a wide verify window share their blocks).
//
// Prefill-class rows (tensor-core kernel): sequences with at least 64 query
// tokens are cut into units of 128 query tokens x one query head.  Units of the
// same KV head are paired (neighbours in key count: the heads of one token tile,
// then adjacent token tiles), so one CTA loads each K/V tile once for two query
// tiles.  One persistent CTA per SM (at most) runs a list of work items of
// equal total cost: whole pairs first, then pieces of the leftover sub-tiles
// cut along their keys, whose partial results a merge combines.
#include <algorithm>
#include <array>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <queue>
#include <vector>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kDecodeWarpsPerSm = 8;
constexpr int kMinBlocksPerWarp = 4;
// Query tokens from which a sequence's rows go to the tensor-core kernel, when
// the caller leaves the choice to the planner (prefill_min_q == 0).
constexpr int kPrefillMinQDefault = 64;
// Relative costs used to give the persistent prefill CTAs equal work: a CTA
// runs a work item's sub-tiles one after the other, each a pass over its key
// tiles, so a pair costs the sum of its sub-tiles' passes: a key tile of one
// sub-tile, and starting a pass (Q load, pipeline fill, epilogue).
constexpr int64_t kTileCost = 8, kPassStartCost = 24;
// CTAs get at least this many key tiles of work.
constexpr int64_t kMinTilesPerCta = 4;

// 0: the default; > 0: that many query tokens; < 0: no sequence (every row on
// the split-KV kernel).
int prefill_threshold(int32_t prefill_min_q) {
  if (prefill_min_q == 0) return kPrefillMinQDefault;
  return prefill_min_q < 0 ? INT_MAX : prefill_min_q;
}

pkv_status check_desc(const pkv_pool_desc *desc, int32_t num_q_heads) {
  if (!desc) return PKV_ERR_NULL;
  if (desc->block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (desc->num_kv_heads < 1 || desc->num_blocks < 0) return PKV_ERR_SHAPE;
  if (num_q_heads < 1 || num_q_heads % desc->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (num_q_heads / desc->num_kv_heads > kRowsPerTile) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

struct Segment {
  int32_t seq, qi0, n_q, h, kb0, nb;  // blocks kb0 .. kb0 + nb - 1
};
struct DUnit {  // a decode row group: n_q tokens from qi0 of seq, reading blocks 0 .. nb-1
  int32_t seq, qi0, n_q, nb;
};
// Shared prefixes shorter than this many blocks stay on the per-warp ranges.
constexpr int32_t kMinSharedBlocks = 8;
// Blocks per 128-key tile of the tensor-core kernel, and the query rows per KV
// head from which a shared prefix goes to it as gathered sub-tiles.
constexpr int32_t kKeyTileBlocks = 128 / kBlockSize;
constexpr int64_t kGatherMinRows = 64;

// The planner's working arrays, kept per host thread so a plan allocates
// nothing once a thread has planned a step of that size.
struct PlanScratch {
  std::vector<std::pair<int32_t, int32_t>> by_first;
  std::vector<Segment> segs;
  std::vector<DUnit> dunits;
  std::vector<Piece> pieces;
  std::vector<int32_t> warp_begin, seg_first, seg_count, seg_of, unit_kb0, shared_len;
  std::vector<int64_t> cut;
  std::vector<MergeGroup> merges;
  std::vector<std::array<int32_t, 3>> sh_ref;  // (unit * hkv + h, item, warp slot)
  std::vector<std::array<int32_t, 2>> sh_list;  // (item, warp slot) grouped by key
  std::vector<int32_t> sh_begin;                // key k: sh_list[sh_begin[k] .. sh_begin[k+1])
  std::vector<int32_t> sh_fill;
  std::vector<std::array<int32_t, 3>> sh_units;
  std::vector<SharedItem> sitems;
};
thread_local PlanScratch t_scratch;

PrefillTile new_tile() {
  PrefillTile t;
  std::memset(&t, 0, sizeof t);
  t.part[0] = t.part[1] = -1;
  t.gather[0] = t.gather[1] = -1;
  return t;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

// lookahead > 0: a plan for `lookahead` further decode steps of the same batch
// (chained decode): every sequence then gains its q_len tokens per step, so the
// decode segments are sized for context + lookahead * q_len; prefill-class
// sequences are not supported there.
// block_tables (host, may be NULL): each warp's first blocks are then written
// into its head.
static pkv_status plan_impl(const int32_t *cu_q_lens, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_q_heads, const pkv_pool_desc *desc,
                            int32_t num_sms, int32_t lookahead, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, int32_t prefill_min_q, void *plan,
                            int64_t plan_capacity, pkv_plan_info *info) {
  if (!info) return PKV_ERR_NULL;
  if (lookahead < 0) return PKV_ERR_RANGE;
  pkv_status st = check_desc(desc, num_q_heads);
  if (st != PKV_OK) return st;
  if (num_seqs < 0) return PKV_ERR_SHAPE;
  if (num_seqs > 0 && (!cu_q_lens || !context_lens)) return PKV_ERR_NULL;
  if (num_sms <= 0) num_sms = device_sm_count();
  if (num_sms <= 0) return PKV_ERR_CUDA;

  const int32_t hkv = desc->num_kv_heads;
  const int32_t group = num_q_heads / hkv;
  const int32_t nq_tile = std::max(1, kRowsPerTile / group);

  // ---- validate; build decode segments and prefill tiles
  if (num_seqs > 0 && cu_q_lens[0] != 0) return PKV_ERR_SHAPE;
  const int min_q_prefill = prefill_threshold(prefill_min_q);
  PlanScratch &S = t_scratch;
  std::vector<Segment> &segs = S.segs;
  std::vector<DUnit> &dunits = S.dunits;
  segs.clear();
  dunits.clear();
  std::vector<PrefillTile> pairs;                 // sub-tile pairs, key range not yet cut
  std::vector<std::array<int32_t, 2>> pair_nt;   // key tiles seen by each sub-tile
  int64_t kv_tokens = 0, total_blocks = 0;
  int32_t max_nb = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t qs64 = (int64_t)cu_q_lens[s + 1] - (int64_t)cu_q_lens[s];
    if (qs64 < 0) return PKV_ERR_SHAPE;
    int32_t qs = (int32_t)qs64, ctx = context_lens[s];
    if (ctx < 0 || qs > ctx) return PKV_ERR_RANGE;
    if (qs == 0) continue;
    kv_tokens += ctx;
    if (lookahead > 0 && qs >= min_q_prefill) return PKV_ERR_UNSUPPORTED;
    const int64_t ctx_plan64 = (int64_t)ctx + (int64_t)lookahead * qs;  // context at the last step
    if (ctx_plan64 > INT32_MAX - kBlockSize) return PKV_ERR_RANGE;
    const int32_t ctx_plan = (int32_t)ctx_plan64;
    max_nb = std::max(max_nb, (ctx_plan + kBlockSize - 1) / kBlockSize);
    if (qs >= min_q_prefill) {
      // units of 128 tokens x 1 query head; within one KV head, sorted by the
      // keys they see, neighbours pair up into one work item (sub-tile 0 sees
      // at least as many keys as sub-tile 1)
      struct Unit {
        int32_t hq, qi0, n_q;
        int64_t keys;
      };
      std::vector<Unit> units;
      for (int32_t h = 0; h < hkv; ++h) {
        units.clear();
        for (int32_t qi0 = qs - 1 - (qs - 1) % kPrefillRows; qi0 >= 0; qi0 -= kPrefillRows) {
          const int32_t n_q = std::min(kPrefillRows, qs - qi0);
          for (int32_t hq = h * group; hq < (h + 1) * group; ++hq)
            units.push_back({hq, qi0, n_q, (int64_t)ctx - qs + qi0 + n_q});
        }
        for (size_t u = 0; u < units.size(); u += 2) {
          PrefillTile t = new_tile();
          t.seq = s;
          t.h = h;
          t.hq[0] = units[u].hq;
          t.qi0[0] = units[u].qi0;
          t.n_q[0] = units[u].n_q;
          if (u + 1 < units.size()) {
            t.hq[1] = units[u + 1].hq;
            t.qi0[1] = units[u + 1].qi0;
            t.n_q[1] = units[u + 1].n_q;
          }
          t.part[0] = t.part[1] = -1;
          pairs.push_back(t);
          pair_nt.push_back({(int32_t)((units[u].keys + kPrefillRows - 1) / kPrefillRows),
                             u + 1 < units.size()
                                 ? (int32_t)((units[u + 1].keys + kPrefillRows - 1) / kPrefillRows)
                                 : 0});
        }
      }
      continue;
    }
    for (int32_t qi0 = 0; qi0 < qs; qi0 += nq_tile) {
      int32_t n_q = std::min(nq_tile, qs - qi0);
      int32_t nb = (ctx_plan - qs + qi0 + n_q - 1) / kBlockSize + 1;
      dunits.push_back({s, qi0, n_q, nb});
    }
  }

  // ---- shared prefixes (needs the host block tables): decode-class sequences
  // whose tables start with the same physical blocks, over blocks every query
  // row of each of them sees in full.  Those blocks are read once per CTA by
  // shared items; the rest of each row group's keys (its suffix) go to the
  // per-warp ranges below.
  std::vector<int32_t> &shared_len = S.shared_len;
  shared_len.assign(num_seqs, 0);
  struct Group {
    std::vector<int32_t> members;
    int32_t len;  // shared blocks handled as shared (whole key tiles when tc)
    bool tc;      // gathered sub-tiles on the tensor-core kernel, else split-KV CTAs
  };
  std::vector<Group> groups;
  if (block_tables && max_blocks_per_seq > 0) {
    // sequences keyed by their first physical block; runs of equal keys are
    // candidate groups (in order of first block, members in sequence order)
    std::vector<std::pair<int32_t, int32_t>> &by_first = S.by_first;
    by_first.clear();
    for (int32_t s = 0; s < num_seqs; ++s) {
      const int32_t qs = cu_q_lens[s + 1] - cu_q_lens[s];
      if (qs <= 0 || qs >= min_q_prefill) continue;
      const int32_t vis = std::min((context_lens[s] - qs + 1) / kBlockSize, max_blocks_per_seq);
      if (vis >= kMinSharedBlocks) by_first.push_back({block_tables[(int64_t)s * max_blocks_per_seq], s});
    }
    std::sort(by_first.begin(), by_first.end());
    std::vector<int32_t> mem;
    for (size_t a = 0, b = 0; a < by_first.size(); a = b) {
      while (b < by_first.size() && by_first[b].first == by_first[a].first) ++b;
      if (b - a < 2) continue;
      mem.clear();
      for (size_t i = a; i < b; ++i) mem.push_back(by_first[i].second);
      int32_t len = INT32_MAX;
      for (int32_t m : mem)
        len = std::min(len, std::min((context_lens[m] - (cu_q_lens[m + 1] - cu_q_lens[m]) + 1) /
                                         kBlockSize, max_blocks_per_seq));
      const int32_t *t0 = block_tables + (int64_t)mem[0] * max_blocks_per_seq;
      for (int32_t kb = 1; kb < len; ++kb)
        for (size_t i = 1; i < mem.size(); ++i)
          if (block_tables[(int64_t)mem[i] * max_blocks_per_seq + kb] != t0[kb]) {
            len = kb;
            break;
          }
      if (len < kMinSharedBlocks) continue;
      int64_t rows = 0;
      for (int32_t m : mem) rows += (int64_t)(cu_q_lens[m + 1] - cu_q_lens[m]) * group;
      const int32_t len_tc = len / kKeyTileBlocks * kKeyTileBlocks;
      const bool tc = lookahead == 0 && len_tc >= kKeyTileBlocks && rows >= kGatherMinRows;
      if (tc) len = len_tc;
      groups.push_back({mem, len, tc});
      for (int32_t m : mem) shared_len[m] = len;
    }
  }
  // ---- shared streams for the split-KV shared-block items: each CTA-path
  // group's prefix (all its members' row groups), and each verify window wider
  // than one row group (its row groups in pairs, over the blocks the pair's first
  // row group sees; the second row group keeps its few later blocks as a
  // suffix).  unit_kb0: where each row group's own (suffix) segment starts.
  struct Stream {
    int32_t seq0, len;
    std::vector<int32_t> units;
  };
  std::vector<Stream> streams;
  std::vector<int32_t> &unit_kb0 = S.unit_kb0;
  unit_kb0.assign(dunits.size(), 0);
  {
    std::vector<int32_t> unit_first(num_seqs, -1);  // decode units are in sequence order
    for (size_t u = dunits.size(); u-- > 0;) unit_first[dunits[u].seq] = (int32_t)u;
    for (size_t u = 0; u < dunits.size(); ++u) unit_kb0[u] = shared_len[dunits[u].seq];
    for (const Group &g : groups) {
      if (g.tc) continue;
      Stream st{g.members[0], g.len, {}};
      for (int32_t m : g.members)
        for (size_t u = unit_first[m]; u < dunits.size() && dunits[u].seq == m; ++u)
          st.units.push_back((int32_t)u);
      streams.push_back(st);
    }
    const size_t n_group_streams = streams.size();
    int64_t window_items = 0;
    for (int32_t sq = 0; sq < num_seqs; ++sq) {
      if (shared_len[sq] > 0 || unit_first[sq] < 0) continue;
      const size_t u0 = unit_first[sq];
      size_t u1 = u0;
      while (u1 < dunits.size() && dunits[u1].seq == sq) ++u1;
      for (size_t u = u0; u + 1 < u1; u += 2) {
        const int32_t len = std::min(dunits[u].nb, dunits[u + 1].nb);
        if (len < kMinSharedBlocks) continue;
        streams.push_back({sq, len, {(int32_t)u, (int32_t)u + 1}});
        window_items += hkv;
      }
    }
    // windows only while one chunk each leaves half the warp slots to the rest
    // (else the shared items alone would take more than a wave)
    if (kSharedRowGroups * window_items * 2 > (int64_t)num_sms * kDecodeWarpsPerSm)
      streams.resize(n_group_streams);
    for (size_t i = n_group_streams; i < streams.size(); ++i)
      for (int32_t u : streams[i].units) unit_kb0[u] = streams[i].len;
  }

  // suffix segments: (row group, KV head) keys past the shared blocks
  std::vector<int32_t> &seg_of = S.seg_of;
  seg_of.assign(dunits.size() * hkv, -1);
  {
    size_t nseg = 0;
    for (size_t u = 0; u < dunits.size(); ++u)
      if (dunits[u].nb > std::min(unit_kb0[u], dunits[u].nb)) nseg += (size_t)hkv;
    segs.resize(nseg);
    Segment *sg = segs.data();
    int32_t *so = seg_of.data();
    int32_t k = 0;
    for (size_t u = 0; u < dunits.size(); ++u) {
      const DUnit du = dunits[u];
      const int32_t kb0 = std::min(unit_kb0[u], du.nb);
      if (du.nb <= kb0) continue;
      for (int32_t h = 0; h < hkv; ++h, ++k) {
        so[u * hkv + h] = k;
        sg[k] = {du.seq, du.qi0, du.n_q, h, kb0, du.nb - kb0};
      }
      total_blocks += (int64_t)hkv * (du.nb - kb0);
    }
  }

  // Both kernels get every SM: the tensor-core kernel's persistent CTAs take one
  // SM each, and the split-KV kernel, which it lets launch once the pool is
  // complete, starts on each SM as soon as that SM's CTA has finished.
  const int32_t pf_sms = num_sms, dec_sms = num_sms;

  // ---- shared-block items: per stream and KV head, its row groups in pairs
  // (a unit); the units' blocks are laid end to end and cut into P equal
  // ranges, one per pair of warps, and a pair's items are the parts of the
  // units its range covers, run one after another (chained through
  // SharedItem::next, its first item at index = pair).  Under the full load of
  // the step a pair streams its blocks at about a single warp's rate (both of
  // its warps attend every block, and a stage is refilled only once both have
  // released it), so P is where P pairs carrying the shared blocks take as long
  // as the slots left over for the independent segments (same-box steps with
  // 4- and 8-token windows, the pair's time per block taken as 3/4, 9/10, 1,
  // 11/10, 5/4 and 3/2 of a warp's: 1 was best).
  const int64_t slots = (int64_t)dec_sms * kDecodeWarpsPerSm;
  std::vector<SharedItem> &sitems = S.sitems;
  sitems.clear();
  int32_t n_pairs = 0;  // heads: sitems[0 .. n_pairs)
  // shared parts of each (decode unit, KV head): (item, warp slot) in key order
  // of the units' blocks, gathered into sh_list below
  std::vector<std::array<int32_t, 3>> &sh_ref = S.sh_ref;
  sh_ref.clear();
  if (!streams.empty()) {
    // the units, in stream order: (stream, KV head, first row group)
    std::vector<std::array<int32_t, 3>> &units = S.sh_units;
    units.clear();
    int64_t sh_blocks = 0;
    for (size_t si = 0; si < streams.size(); ++si) {
      const Stream &st = streams[si];
      for (int32_t h = 0; h < hkv; ++h)
        for (size_t i0 = 0; i0 < st.units.size(); i0 += kSharedRowGroups) {
          units.push_back({(int32_t)si, h, (int32_t)i0});
          sh_blocks += st.len;
        }
    }
    // independent load in block steps of one warp: its blocks plus 3 per segment
    const int64_t ind = total_blocks + 3 * (int64_t)segs.size();
    const int64_t max_pairs = std::max<int64_t>(1, slots / kSharedRowGroups - (ind > 0 ? 1 : 0));
    int64_t np2 = ind > 0 ? (sh_blocks * slots) / (ind + 2 * sh_blocks) : max_pairs;
    np2 = std::max<int64_t>(1, std::min<int64_t>({np2, max_pairs, sh_blocks / kMinBlocksPerWarp}));
    // whole CTAs
    n_pairs = (int32_t)(np2 + (np2 % kSharedItemsPerCta ? kSharedItemsPerCta - np2 % kSharedItemsPerCta : 0));
    // a pair's range starts at most one item beyond the units it covers
    sitems.reserve((size_t)n_pairs + units.size() + (size_t)n_pairs);
    sitems.resize(n_pairs);
    std::memset(sitems.data(), 0, (size_t)n_pairs * sizeof(SharedItem));
    for (int32_t k = 0; k < n_pairs; ++k) sitems[k].next = -1;  // empty (n_rg == 0) until it gets an item
    size_t u = 0;
    int64_t u_off = 0;  // first position of unit u
    for (int32_t k = 0; k < n_pairs; ++k) {
      const int64_t lo = sh_blocks * k / n_pairs, hi = sh_blocks * (k + 1) / n_pairs;
      int32_t prev = -1;
      for (int64_t a = lo; a < hi;) {
        while (u_off + streams[units[u][0]].len <= a) u_off += streams[units[u++][0]].len;
        const Stream &st = streams[units[u][0]];
        const int64_t e = std::min<int64_t>(hi, u_off + st.len);
        SharedItem it;
        std::memset(&it, 0, sizeof it);
        it.seq0 = st.seq0;
        it.h = units[u][1];
        it.kb_begin = (int32_t)(a - u_off);
        it.kb_end = (int32_t)(e - u_off);
        const size_t i0 = (size_t)units[u][2];
        it.n_rg = (int32_t)std::min<size_t>(kSharedRowGroups, st.units.size() - i0);
        it.next = -1;
        const int32_t idx = prev < 0 ? k : (int32_t)sitems.size();
        for (int32_t w = 0; w < it.n_rg; ++w) {
          const DUnit &du = dunits[st.units[i0 + w]];
          it.rg[w].seq = du.seq;
          it.rg[w].qi0 = du.qi0;
          it.rg[w].n_q = du.n_q;
          it.rg[w].part = -1;
          it.rg[w].q_row0 = cu_q_lens[du.seq] + du.qi0;
          sh_ref.push_back({(int32_t)((size_t)st.units[i0 + w] * hkv + it.h), idx, w});
        }
        if (prev < 0)
          sitems[k] = it;
        else
          sitems.push_back(it);
        if (prev >= 0) sitems[prev].next = idx;
        prev = idx;
        a = e;
      }
    }
  }
  // sh_ref grouped by key (a counting sort; each key keeps its creation order,
  // i.e. its blocks' order)
  std::vector<std::array<int32_t, 2>> &sh_list = S.sh_list;
  std::vector<int32_t> &sh_begin = S.sh_begin;
  if (!sh_ref.empty()) {
    const size_t nkeys = dunits.size() * (size_t)hkv;
    sh_begin.assign(nkeys + 1, 0);
    for (const auto &rf : sh_ref) ++sh_begin[rf[0] + 1];
    for (size_t k = 0; k < nkeys; ++k) sh_begin[k + 1] += sh_begin[k];
    sh_list.resize(sh_ref.size());
    std::vector<int32_t> &fill = S.sh_fill;  // per-key fill positions
    fill.assign(sh_begin.begin(), sh_begin.end() - 1);
    for (const auto &rf : sh_ref) sh_list[fill[rf[0]]++] = {rf[1], rf[2]};
  }
  const int64_t shared_slots = (int64_t)n_pairs * kSharedRowGroups;

  // ---- gathered sub-tiles (tc groups): per group and KV head, the members'
  // query tokens in sub-tiles of up to 128 / G tokens (G rows each); every
  // sub-tile is cut along the prefix's key tiles into nc equal chunks, one work
  // item each, nc chosen so the items about fill their share of the SMs (at
  // least 2 key tiles each)
  std::vector<GatherRow> gather;          // part0 filled once partial slots are known
  std::vector<int32_t> gather_uh;         // (decode unit * hkv + KV head) of each entry
  std::vector<PrefillTile> casc_items;    // already cut along keys
  std::vector<int32_t> unit_casc(dunits.size(), 0);  // key chunks of each unit's prefix
  {
    struct Sub {
      int32_t first, n;
    };
    struct CPair {
      int32_t gi, h;
      Sub sub[2];
      int32_t nsub;
    };
    std::vector<CPair> cpairs;
    const int32_t tok_per_sub = std::max(1, kPrefillRows / group);
    std::vector<int32_t> unit_first(num_seqs, -1);  // decode units are in sequence order
    for (size_t u = dunits.size(); u-- > 0;) unit_first[dunits[u].seq] = (int32_t)u;
    for (size_t gi = 0; gi < groups.size(); ++gi) {
      const Group &g = groups[gi];
      if (!g.tc) continue;
      std::vector<std::array<int32_t, 3>> toks;  // (unit, packed token, row of its first head)
      for (int32_t m : g.members)
        for (size_t u = unit_first[m]; u < dunits.size() && dunits[u].seq == m; ++u)
          for (int32_t i = 0; i < dunits[u].n_q; ++i)
            toks.push_back({(int32_t)u, cu_q_lens[m] + dunits[u].qi0 + i, i * group});
      for (int32_t h = 0; h < hkv; ++h) {
        std::vector<Sub> subs;
        for (size_t t0 = 0; t0 < toks.size(); t0 += tok_per_sub) {
          const int32_t n = (int32_t)std::min<size_t>(tok_per_sub, toks.size() - t0);
          subs.push_back({(int32_t)gather.size(), n});
          for (int32_t i = 0; i < n; ++i) {
            const auto &tk = toks[t0 + i];
            gather.push_back({tk[1], -1, tk[2], 0});
            gather_uh.push_back(tk[0] * hkv + h);
          }
        }
        // one sub-tile per item: a CTA's two sub-tiles would run as two
        // passes over the same keys, each paying its start and its partial
        // epilogue (same box: shared-prefix verify 50.7 -> 45.4 us, MTP draft
        // 45.3 -> 44.8 us against pairs of sub-tiles)
        for (size_t k = 0; k < subs.size(); ++k) {
          CPair cp;
          cp.gi = (int32_t)gi;
          cp.h = h;
          cp.sub[0] = subs[k];
          cp.sub[1] = Sub{-1, 0};
          cp.nsub = 1;
          cpairs.push_back(cp);
        }
      }
    }
    if (!cpairs.empty()) {
      // The items take a share of the SMs; the split-KV kernel streams the
      // step's own blocks on the rest meanwhile (only there: see the warp
      // count below).  Share = prefix tile passes / (tile passes + streamed
      // block-heads / 16), at least 7/16: a tile pass weighed as 16
      // block-heads and that floor put both shared-prefix workloads at their
      // measured optimum (same box, one chunk per sub-tile fewer and one more:
      // shared-prefix verify 64 of 152 SMs, 45.4 us against 60.1 at 32 and
      // 55.8 at 96; MTP draft 64, 44.8 us against 45.4 at 48 and 49.0 at
      // 80).  Integer arithmetic, so every host plans alike.
      int64_t pf_work = 0;
      for (const CPair &cp : cpairs) pf_work += (int64_t)cp.nsub * (groups[cp.gi].len / kKeyTileBlocks);
      const int64_t ncp = (int64_t)cpairs.size();
      int64_t num = 16 * pf_work, den = 16 * pf_work + total_blocks;  // share = num / den
      if (16 * num < 7 * den) {
        num = 7;
        den = 16;
      }
      const int64_t want = std::max<int64_t>(1, (2 * num * pf_sms + den * ncp) / (2 * den * ncp));
      for (const CPair &cp : cpairs) {
        const Group &g = groups[cp.gi];
        const int32_t kt = g.len / kKeyTileBlocks;
        const int32_t nc = (int32_t)std::max<int64_t>(1, std::min<int64_t>(want, kt / 2));
        for (int32_t m : g.members)
          for (size_t u = unit_first[m]; u < dunits.size() && dunits[u].seq == m; ++u)
            unit_casc[u] = nc;
        for (int32_t c = 0; c < nc; ++c) {
          PrefillTile t = new_tile();
          t.seq = g.members[0];
          t.h = cp.h;
          t.kt0 = (int32_t)((int64_t)kt * c / nc);
          t.kt1 = (int32_t)((int64_t)kt * (c + 1) / nc);
          for (int x = 0; x < cp.nsub; ++x) {
            t.hq[x] = cp.h * group;
            t.n_q[x] = cp.sub[x].n;
            t.gather[x] = cp.sub[x].first;
            t.part[x] = c;
            // consecutive packed tokens: one q box for the whole sub-tile
            bool run = true;
            for (int32_t i = 1; i < cp.sub[x].n && run; ++i)
              run = gather[cp.sub[x].first + i].q_tok == gather[cp.sub[x].first].q_tok + i;
            if (run) {
              t.runs |= 1 << x;
              t.qi0[x] = gather[cp.sub[x].first].q_tok;
            }
          }
          casc_items.push_back(t);
        }
      }
    }
  }

  // ---- cut the concatenated suffix blocks into equal-cost warp ranges
  const int64_t avail = std::max<int64_t>(slots - shared_slots, 1);
  int64_t nw64 = (total_blocks + kMinBlocksPerWarp - 1) / kMinBlocksPerWarp;
  nw64 = std::min<int64_t>(nw64, avail);
  // Behind a tensor-core prefill whose persistent CTAs take every SM (enough
  // key tiles for all of them) the split-KV CTAs start one after another, in
  // index order, as those CTAs exit, and a CTA's few blocks take a
  // latency-bound ~8 us whatever their number: half the warp slots, on the SMs
  // freed first, finish with the prefill instead of ~9 us after it
  // (agent-shaped step, same box: 146.5 -> 144.3 us; 2/3 and 2/5 of the slots
  // in between, a quarter 149.7).  A smaller prefill leaves SMs free from the
  // start and keeps every slot.
  if (!pairs.empty()) {
    int64_t pf_tiles = 0;
    for (const auto &nt : pair_nt) pf_tiles += nt[0] + nt[1];
    if (pf_tiles >= (int64_t)pf_sms * kMinTilesPerCta)
      nw64 = std::min<int64_t>(nw64, std::max<int64_t>(1, avail / 2));
  }
  // With gathered prefix items as the step's only tensor-core work, the
  // lowest-index split-KV CTAs start at once on the SMs the items leave free
  // and stream while the items run; the others could start only as the items'
  // CTAs exit, and then need several latency-bound us for however few blocks.
  // So the split-KV work goes to the free SMs' warp slots alone (same box:
  // shared-prefix verify 55.6 -> 49.7 us, MTP draft 49.5 -> 47.3 us against
  // the same warps taking 4 times a late warp's share, 54.0 / 49.1 at 8 times).
  if (pairs.empty() && !casc_items.empty() && (int64_t)casc_items.size() < dec_sms)
    nw64 = std::min<int64_t>(nw64, std::max<int64_t>(1, (dec_sms - (int64_t)casc_items.size()) *
                                                            kDecodeWarpsPerSm));
  // Small steps: when every segment fits a warp slot and the longest is within a
  // few blocks of the equal share, one warp per whole segment runs about as long
  // as the equal-cost cut and needs no partials or merge launch.
  int32_t max_seg = 0;
  for (const Segment &g : segs) max_seg = std::max(max_seg, g.nb);
  const bool whole_segments =
      !segs.empty() && (int64_t)segs.size() <= avail &&
      max_seg <= std::max<int64_t>(2 * kMinBlocksPerWarp,
                                   (total_blocks + avail - 1) / avail + kMinBlocksPerWarp);
  if (whole_segments) nw64 = (int64_t)segs.size();
  const int32_t num_warps = total_blocks > 0 ? (int32_t)std::max<int64_t>(nw64, 1) : 0;
  std::vector<int32_t> &warp_begin = S.warp_begin;
  warp_begin.assign(num_warps + 1, 0);
  // Pieces go straight into the caller's plan buffer when it surely holds them
  // (their offset depends only on the warp count; a range adds at most one
  // piece beyond its segments), else into a scratch array copied at the end.
  const int64_t off_pieces = (int64_t)sizeof(PlanHeader) + align_up(4ll * (num_warps + 1), 32) +
                             (int64_t)num_warps * (int64_t)sizeof(WarpHead);
  const int64_t max_pieces = (int64_t)segs.size() + num_warps;
  const bool pieces_in_plan =
      plan && plan_capacity >= off_pieces + max_pieces * (int64_t)sizeof(Piece);
  if (!pieces_in_plan) S.pieces.resize((size_t)max_pieces);
  Piece *const pieces =
      pieces_in_plan ? reinterpret_cast<Piece *>(static_cast<char *>(plan) + off_pieces)
                     : S.pieces.data();
  int32_t npieces = 0;
  // each segment's pieces are consecutive: its first one and how many
  std::vector<int32_t> &seg_first = S.seg_first, &seg_count = S.seg_count;
  seg_first.assign(segs.size(), -1);
  seg_count.assign(segs.size(), 0);
  {
    // Equal cost, not equal blocks: a block costs kBlockCost and starting a
    // segment (its q rows and lengths, a fresh table window) costs kPieceCost, so
    // a warp whose range crosses into another segment gets fewer blocks.  Block
    // i of segment k sits at cost position start_k + kPieceCost + kBlockCost*i
    // (+ half a block) and goes to the warp whose equal share of the total cost
    // holds that position; the ranges stay contiguous in the block stream.  With
    // at least kMinBlocksPerWarp blocks per warp every share holds a block.
    constexpr int64_t kBlockCost = 2, kPieceCost = 6;
    const int64_t total_cost = kBlockCost * total_blocks + kPieceCost * (int64_t)segs.size();
    std::vector<int64_t> &cut = S.cut;  // first block of each warp
    cut.assign(num_warps + 1, total_blocks);
    cut[0] = 0;
    if (whole_segments) {
      int64_t blk = 0;
      for (int32_t w = 0; w < num_warps; ++w) {
        cut[w] = blk;
        blk += segs[w].nb;
      }
    } else {
      // warp w >= 1 starts at the first block whose midpoint m satisfies
      // m * num_warps >= w * total_cost, i.e. m >= T(w) = ceil(w * total_cost /
      // num_warps); the midpoints of a segment starting at cost c are c +
      // kPieceCost + kBlockCost * i + kBlockCost / 2.  w * total_cost /
      // num_warps is carried from warp to warp as a quotient and remainder, so
      // the whole cut takes no division per warp or per segment.
      static_assert(kBlockCost == 2, "the block index below halves a cost distance");
      const int64_t nwd = std::max<int64_t>(num_warps, 1);
      const int64_t dq = total_cost / nwd, dr = total_cost % nwd;
      int64_t tq = dq, tr = dr;  // w * total_cost = tq * num_warps + tr, 0 <= tr < num_warps
      int32_t w = 1;
      int64_t cost = 0, blk = 0;
      for (const Segment &g : segs) {
        const int64_t first_mid = cost + kPieceCost + kBlockCost / 2;
        const int64_t last_mid = first_mid + kBlockCost * (g.nb - 1);
        while (w < num_warps) {
          const int64_t t = tq + (tr > 0 ? 1 : 0);  // T(w)
          if (last_mid < t) break;
          int64_t i = t > first_mid ? (t - first_mid + 1) >> 1 : 0;  // ceil((t - first_mid) / 2)
          if (i > g.nb - 1) i = g.nb - 1;
          cut[w++] = blk + i;
          tq += dq;
          tr += dr;
          if (tr >= nwd) {
            ++tq;
            tr -= nwd;
          }
        }
        cost += kPieceCost + kBlockCost * g.nb;
        blk += g.nb;
      }
      while (w < num_warps) cut[w++] = total_blocks;
    }
    size_t k = 0;
    int64_t seg_off = 0;  // global block offset of segment k
    const Segment *sg = segs.data();
    const int64_t *ct = cut.data();
    int32_t *wb = warp_begin.data(), *sf = seg_first.data(), *sc = seg_count.data();
    int32_t np = 0;
    for (int32_t w = 0; w < num_warps; ++w) {
      wb[w] = np;
      int64_t a = ct[w];
      const int64_t b = ct[w + 1];
      while (a < b) {
        while (seg_off + sg[k].nb <= a) seg_off += sg[k++].nb;
        const Segment g = sg[k];
        const int64_t e = std::min<int64_t>(b, seg_off + g.nb);
        pieces[np] = {g.seq, g.qi0, g.n_q, g.h, g.kb0 + (int32_t)(a - seg_off),
                      g.kb0 + (int32_t)(e - seg_off), -1, cu_q_lens[g.seq] + g.qi0};
        if (sf[k] < 0) sf[k] = np;
        ++sc[k];
        ++np;
        a = e;
      }
    }
    npieces = np;
    wb[num_warps] = npieces;
  }
  // partial slots: every (decode unit, KV head) result whose keys are split over
  // several parts (shared-prefix chunks and suffix pieces) gets one slot per part
  // and a merge group; a result in one part is written directly
  std::vector<MergeGroup> &merges = S.merges;
  merges.clear();
  int32_t parts = 0;
  int32_t merge_rows = 0;  // rows of the largest decode merge group
  {
    // gathered prefix chunks always write partials: their unit gets a merge
    // group even when nothing else splits it
    std::vector<int32_t> casc_part0(gather.empty() ? 0 : dunits.size() * hkv, -1);
    merges.resize(dunits.size() * (size_t)hkv);  // at most one group per (unit, KV head)
    MergeGroup *mg = merges.data();
    const int32_t *so = seg_of.data(), *sf = seg_first.data(), *sc = seg_count.data();
    size_t nm = 0;
    for (size_t u = 0; u < dunits.size(); ++u) {
      const DUnit du = dunits[u];
      const int32_t nc = unit_casc[u];
      for (int32_t h = 0; h < hkv; ++h) {
        const size_t key = u * hkv + h;
        const int32_t sh0 = sh_ref.empty() ? 0 : sh_begin[key];
        const int32_t sh1 = sh_ref.empty() ? 0 : sh_begin[key + 1];
        const int32_t k = so[u * hkv + h];
        const int32_t np = k >= 0 ? sc[k] : 0;
        const int32_t total = nc + (sh1 - sh0) + np;
        if (total <= 1 && nc == 0) continue;
        mg[nm++] = {du.seq, du.qi0, du.n_q, h, parts, total, 0, cu_q_lens[du.seq] + du.qi0};
        merge_rows = std::max(merge_rows, du.n_q * group);
        if (!casc_part0.empty()) casc_part0[u * hkv + h] = nc > 0 ? parts : -1;
        parts += nc;
        for (int32_t t = sh0; t < sh1; ++t) sitems[sh_list[t][0]].rg[sh_list[t][1]].part = parts++;
        Piece *pc = pieces + (k >= 0 ? sf[k] : 0);
        for (int32_t t = 0; t < np; ++t) pc[t].part = parts++;
      }
    }
    merges.resize(nm);
    for (size_t i = 0; i < gather.size(); ++i) gather[i].part0 = casc_part0[gather_uh[i]];
  }
  // ---- prefill work per persistent CTA (at most one per SM), equal cost:
  //  0. the gathered prefix items (already cut along keys), largest first, each
  //     into the least-loaded CTA;
  //  1. whole pairs, largest first, each into the least-loaded CTA that stays
  //     within the per-CTA target;
  //  2. the pairs left over are split into their sub-tiles, whose key tiles are
  //     laid end to end and cut at the CTAs' remaining capacities.  A sub-tile
  //     cut there gets one partial slot per piece and a merge group (kind 1).
  std::vector<PrefillTile> ptiles;
  std::vector<int32_t> pf_begin;
  std::vector<MergeGroup> pmerges;
  int32_t pparts = 0;
  int32_t n_pf_ctas = 0;
  if (!pairs.empty() || !casc_items.empty()) {
    auto pair_cost = [&](size_t pi) {
      const int64_t nt0 = pair_nt[pi][0], nt1 = pair_nt[pi][1];
      return kPassStartCost * (nt1 > 0 ? 2 : 1) + kTileCost * (nt0 + nt1);
    };
    auto item_cost = [&](const PrefillTile &t) {
      return (kPassStartCost + kTileCost * (t.kt1 - t.kt0)) * (t.n_q[1] > 0 ? 2 : 1);
    };
    int64_t total = 0, ntiles = 0;
    for (size_t pi = 0; pi < pairs.size(); ++pi) {
      total += pair_cost(pi);
      ntiles += pair_nt[pi][0] + pair_nt[pi][1];
    }
    for (const PrefillTile &t : casc_items) {
      total += item_cost(t);
      ntiles += (t.kt1 - t.kt0) * (t.n_q[1] > 0 ? 2 : 1);
    }
    n_pf_ctas = (int32_t)std::max<int64_t>(
        1, std::min<int64_t>(pf_sms, std::max<int64_t>(ntiles / kMinTilesPerCta,
                                                        (int64_t)casc_items.size())));
    const int64_t target = (total + n_pf_ctas - 1) / n_pf_ctas;
    std::vector<size_t> order(pairs.size());
    for (size_t i = 0; i < order.size(); ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](size_t x, size_t y) { return pair_cost(x) > pair_cost(y); });
    std::vector<int64_t> load(n_pf_ctas, 0);
    // (CTA, item) in assignment order; grouped by CTA at the end
    std::vector<std::pair<int32_t, PrefillTile>> assigned;
    assigned.reserve(casc_items.size() + 2 * pairs.size());
    // least-loaded CTA first (lowest index among equals): a min-heap of (load, CTA)
    std::priority_queue<std::pair<int64_t, int32_t>, std::vector<std::pair<int64_t, int32_t>>,
                        std::greater<std::pair<int64_t, int32_t>>>
        least;
    for (int32_t b = 0; b < n_pf_ctas; ++b) least.push({0, b});
    {
      std::vector<size_t> corder(casc_items.size());
      for (size_t i = 0; i < corder.size(); ++i) corder[i] = i;
      std::stable_sort(corder.begin(), corder.end(), [&](size_t x, size_t y) {
        return item_cost(casc_items[x]) > item_cost(casc_items[y]);
      });
      for (size_t ci : corder) {
        const int32_t best = least.top().second;
        least.pop();
        load[best] += item_cost(casc_items[ci]);
        least.push({load[best], best});
        assigned.push_back({best, casc_items[ci]});
      }
    }
    std::vector<size_t> leftover;
    for (size_t pi : order) {
      // the least-loaded CTA takes the pair if it stays within the target (then
      // no CTA can)
      const int64_t pc = pair_cost(pi);
      const int32_t best = least.top().second;
      if (load[best] + pc > target) {
        leftover.push_back(pi);
        continue;
      }
      least.pop();
      load[best] += pc;
      least.push({load[best], best});
      PrefillTile t = pairs[pi];
      t.kt0 = 0;
      t.kt1 = pair_nt[pi][0];
      t.part[0] = t.part[1] = -1;
      assigned.push_back({best, t});
    }
    // leftover sub-tiles, cut at the remaining capacities (CTA order)
    struct Sub {
      size_t pi;
      int x;
    };
    std::vector<Sub> subs;
    int64_t rest = 0;
    for (size_t pi : leftover)
      for (int x = 0; x < 2; ++x)
        if (pair_nt[pi][x] > 0) {
          subs.push_back({pi, x});
          rest += kPassStartCost + kTileCost * pair_nt[pi][x];
        }
    if (!subs.empty()) {
      std::vector<int64_t> room(n_pf_ctas), room_end(n_pf_ctas);
      int64_t room_total = 0;
      for (int32_t b = 0; b < n_pf_ctas; ++b) {
        room[b] = std::max<int64_t>(0, target - load[b]);
        room_total += room[b];
      }
      // CTA b takes the part of the stream [room_end[b-1], room_end[b]) scaled
      // to the stream's total
      int64_t acc = 0;
      for (int32_t b = 0; b < n_pf_ctas; ++b) {
        acc += room[b];
        room_end[b] = room_total > 0 ? acc * rest / room_total : (int64_t)(b + 1) * rest / n_pf_ctas;
      }
      int64_t cost = 0;
      int32_t cta = 0;
      std::vector<std::array<int32_t, 3>> pcs;  // (cta, j0, j1) of one sub-tile
      for (const Sub &u : subs) {
        const PrefillTile &src = pairs[u.pi];
        const int32_t nt = pair_nt[u.pi][u.x];
        cost += kPassStartCost;
        pcs.clear();
        for (int32_t j = 0; j < nt; ++j) {
          const int64_t mid = cost + kTileCost / 2;
          while (cta < n_pf_ctas - 1 && mid >= room_end[cta]) ++cta;
          cost += kTileCost;
          if (pcs.empty() || pcs.back()[0] != cta)
            pcs.push_back({cta, j, j + 1});
          else
            pcs.back()[2] = j + 1;
        }
        int32_t part0 = -1;
        if (pcs.size() > 1) {
          part0 = pparts;
          MergeGroup m;
          std::memset(&m, 0, sizeof m);
          m.seq = src.seq;
          m.qi0 = src.qi0[u.x];
          m.q_row0 = cu_q_lens[src.seq] + src.qi0[u.x];
          m.n_q = src.n_q[u.x];
          m.h = src.hq[u.x];
          m.part0 = pparts;
          m.nsplit = (int32_t)pcs.size();
          m.kind = 1;
          pmerges.push_back(m);
          pparts += (int32_t)pcs.size();
        }
        for (size_t k = 0; k < pcs.size(); ++k) {
          PrefillTile t = new_tile();
          t.seq = src.seq;
          t.h = src.h;
          t.hq[0] = src.hq[u.x];
          t.qi0[0] = src.qi0[u.x];
          t.n_q[0] = src.n_q[u.x];
          t.kt0 = pcs[k][1];
          t.kt1 = pcs[k][2];
          t.part[0] = part0 >= 0 ? part0 + (int32_t)k : -1;
          t.part[1] = -1;
          assigned.push_back({pcs[k][0], t});
        }
      }
    }
    // CTAs the assignment left without work are dropped (a CTA always has at
    // least one item)
    std::vector<int32_t> slot(n_pf_ctas + 1, 0);  // items per CTA, then each kept CTA's first slot
    for (const auto &a : assigned) ++slot[a.first];
    int32_t kept = 0, at = 0;
    pf_begin.clear();
    for (int32_t b = 0; b < n_pf_ctas; ++b) {
      const int32_t cnt = slot[b];
      slot[b] = at;
      if (cnt > 0) {
        pf_begin.push_back(at);
        ++kept;
      }
      at += cnt;
    }
    pf_begin.push_back(at);
    n_pf_ctas = kept;
    ptiles.resize(assigned.size());
    for (const auto &a : assigned) ptiles[slot[a.first]++] = a.second;  // stable within a CTA
  }
  for (const MergeGroup &m : pmerges) merges.push_back(m);  // after the decode groups

  // ---- sizes
  const PlanOffsets off =
      plan_offsets(num_warps, npieces, (int32_t)merges.size(),
                   (int32_t)sitems.size(), (int32_t)ptiles.size(), n_pf_ctas, (int32_t)gather.size());
  std::memset(info, 0, sizeof *info);
  info->num_seqs = num_seqs;
  info->num_q_heads = num_q_heads;
  info->num_kv_heads = hkv;
  info->head_dim = desc->head_dim;
  info->total_q = num_seqs > 0 ? cu_q_lens[num_seqs] : 0;
  info->num_decode_warps = num_warps;
  info->num_decode_pieces = npieces;
  info->num_merge_groups = (int32_t)merges.size();
  info->num_partials = parts;
  info->num_prefill_tiles = (int32_t)ptiles.size();
  info->num_prefill_ctas = n_pf_ctas;
  info->num_prefill_partials = pparts;
  info->num_prefill_merges = (int32_t)pmerges.size();
  info->num_kernels = (num_warps > 0 || !sitems.empty() ? 1 : 0) + (merges.empty() ? 0 : 1) +
                      (ptiles.empty() ? 0 : 1);
  info->num_shared_ctas = n_pairs / kSharedItemsPerCta;
  info->num_shared_items = (int32_t)sitems.size();
  info->num_gather_rows = (int32_t)gather.size();
  info->merge_rows = merge_rows;
  info->max_blocks_needed = max_nb;
  info->kv_tokens = kv_tokens;
  // blocks the split-KV kernel attends, each once: every decode-class sequence's
  // blocks past its shared part, plus each CTA-path group's shared blocks
  int64_t dec_blocks = 0, gather_pairs = 0;
  {
    std::vector<int32_t> seq_nb(num_seqs, 0);
    for (const DUnit &du : dunits) seq_nb[du.seq] = std::max(seq_nb[du.seq], du.nb);
    for (int32_t s = 0; s < num_seqs; ++s)
      if (seq_nb[s] > shared_len[s]) dec_blocks += (int64_t)hkv * (seq_nb[s] - shared_len[s]);
    for (const Group &g : groups)
      if (!g.tc) dec_blocks += (int64_t)hkv * g.len;
  }
  for (const PrefillTile &t : casc_items)
    gather_pairs += (int64_t)(t.n_q[0] + t.n_q[1]) * group * (t.kt1 - t.kt0) * 128;
  info->decode_blocks = dec_blocks;
  info->gather_pairs = gather_pairs;
  info->plan_bytes = off.total;
  info->workspace_bytes = ws_total_bytes(parts, pparts, desc->head_dim);
  info->lookahead = lookahead;

  if (!plan) return PKV_OK;
  if (plan_capacity < info->plan_bytes) return PKV_ERR_WORKSPACE;
  char *p = static_cast<char *>(plan);
  // every section below is written whole; only the alignment padding after
  // the two offset arrays is cleared
  {
    const int64_t wb_end = off.warp_begin + (int64_t)warp_begin.size() * 4;
    std::memset(p + wb_end, 0, (size_t)(off.warp_head - wb_end));
    const int64_t pb_end = off.prefill_begin + (int64_t)pf_begin.size() * 4;
    if (off.prefill > pb_end) std::memset(p + pb_end, 0, (size_t)(off.prefill - pb_end));
  }
  PlanHeader h;
  std::memset(&h, 0, sizeof h);
  h.magic = kPlanMagic;
  h.num_seqs = num_seqs;
  h.num_q_heads = num_q_heads;
  h.num_kv_heads = hkv;
  h.head_dim = desc->head_dim;
  h.total_q = info->total_q;
  h.num_decode_warps = num_warps;
  h.num_decode_pieces = info->num_decode_pieces;
  h.num_merge_groups = info->num_merge_groups;
  h.num_partials = parts;
  h.num_prefill_tiles = info->num_prefill_tiles;
  h.max_blocks_needed = max_nb;
  h.reserved[0] = (int32_t)gather.size();
  std::memcpy(p, &h, sizeof h);
  std::memcpy(p + off.warp_begin, warp_begin.data(), warp_begin.size() * sizeof(int32_t));
  WarpHead *heads = reinterpret_cast<WarpHead *>(p + off.warp_head);
  for (int32_t w = 0; w < num_warps; ++w) {
    WarpHead &wh = heads[w];
    if (warp_begin[w] >= warp_begin[w + 1]) {  // a warp without blocks
      std::memset(&wh, 0, sizeof wh);
      wh.first.seq = -1;
      for (int i = 0; i < 4; ++i) wh.blk[i] = -1;
      continue;
    }
    wh.first = pieces[warp_begin[w]];
    for (int i = 0; i < 4; ++i) {
      const int32_t kb = wh.first.kb_begin + i;
      wh.blk[i] = -1;
      if (i < kHeadBlocks && block_tables && kb < wh.first.kb_end && kb < max_blocks_per_seq)
        wh.blk[i] = block_tables[(int64_t)wh.first.seq * max_blocks_per_seq + kb];
    }
  }
  if (npieces > 0 && !pieces_in_plan)
    std::memcpy(p + off.pieces, pieces, (size_t)npieces * sizeof(Piece));
  if (!merges.empty())
    std::memcpy(p + off.merges, merges.data(), merges.size() * sizeof(MergeGroup));
  if (!sitems.empty())
    std::memcpy(p + off.shared, sitems.data(), sitems.size() * sizeof(SharedItem));
  if (!ptiles.empty()) {
    std::memcpy(p + off.prefill_begin, pf_begin.data(), pf_begin.size() * sizeof(int32_t));
    std::memcpy(p + off.prefill, ptiles.data(), ptiles.size() * sizeof(PrefillTile));
  }
  if (!gather.empty())
    std::memcpy(p + off.gather, gather.data(), gather.size() * sizeof(GatherRow));
  return PKV_OK;
}

// The planner's host scratch grows with the step; no C++ exception (a failed
// allocation) leaves the C ABI: it becomes PKV_ERR_HOST_MEMORY.
static pkv_status plan_guarded(const int32_t *cu_q_lens, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, const pkv_pool_desc *desc,
                               int32_t num_sms, int32_t lookahead, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, int32_t prefill_min_q, void *plan,
                               int64_t plan_capacity, pkv_plan_info *info) {
  try {
    return plan_impl(cu_q_lens, context_lens, num_seqs, num_q_heads, desc, num_sms, lookahead,
                     block_tables, max_blocks_per_seq, prefill_min_q, plan, plan_capacity, info);
  } catch (...) {
    return PKV_ERR_HOST_MEMORY;
  }
}

extern "C" pkv_status pkv_plan_step_ex(const int32_t *cu_q_lens, const int32_t *context_lens,
                                       int32_t num_seqs, int32_t num_q_heads,
                                       const pkv_pool_desc *desc, int32_t num_sms, int32_t steps,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       int32_t prefill_min_q, void *plan, int64_t plan_capacity,
                                       pkv_plan_info *info) {
  if (steps < 1) return PKV_ERR_RANGE;
  if (block_tables && max_blocks_per_seq < 0) return PKV_ERR_SHAPE;
  return plan_guarded(cu_q_lens, context_lens, num_seqs, num_q_heads, desc, num_sms, steps - 1,
                      block_tables, max_blocks_per_seq, prefill_min_q, plan, plan_capacity, info);
}

extern "C" pkv_status pkv_plan_step(const int32_t *cu_q_lens, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    const pkv_pool_desc *desc, int32_t num_sms, void *plan,
                                    int64_t plan_capacity, pkv_plan_info *info) {
  return plan_guarded(cu_q_lens, context_lens, num_seqs, num_q_heads, desc, num_sms, 0, nullptr, 0,
                      0, plan, plan_capacity, info);
}

extern "C" pkv_status pkv_plan_decode_chain(const int32_t *cu_q_lens, const int32_t *context_lens,
                                            int32_t num_seqs, int32_t num_q_heads,
                                            const pkv_pool_desc *desc, int32_t num_sms,
                                            int32_t steps, void *plan, int64_t plan_capacity,
                                            pkv_plan_info *info) {
  return pkv_plan_step_ex(cu_q_lens, context_lens, num_seqs, num_q_heads, desc, num_sms, steps,
                          nullptr, 0, 0, plan, plan_capacity, info);
}
