// Split-KV paged attention for decode-class rows, plus the LSE merge.
//
// What it computes is the packed varlen attention of the vllm-metal page
// ("Replacing attention, reusing the rest"): every query row attends over the
// keys of its sequence visible under the causal rule, keys read from pool
// blocks through the sequence's block table.  The page's own kernel is a Metal
// port of a Triton kernel; this is a GB300 design:
//
//  * The host planner lays every (row group, KV head) segment's blocks end to
//    end and cuts them into equal contiguous ranges, one per warp (8 warps per
//    SM, one wave).  A warp's range crosses one or more segments; each piece is
//    finished in registers and written either as final output or as an fp32
//    partial.  No CTA-wide barrier, no shared-memory merge.
//  * A row group is n_q query tokens x all `group` query heads sharing the KV
//    head (<= 16 rows = one m16 MMA tile), so each KV block read from HBM serves
//    every query head of the group (GQA sharing).
//  * Each warp owns a private NSTAGE-deep ring in shared memory.  Lane 0 issues
//    the K and V boxes of the next block of the warp's stream with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle) against the stage's mbarrier; the
//    stream runs on across piece boundaries, so HBM requests never stop at a
//    segment edge.
//  * Q K^T and P V run on mma.sync m16n8k16 (bf16 in, fp32 accumulate) with
//    fragments read straight from the swizzled tiles: the head_dim index is
//    permuted identically in the Q and K fragments so each lane reads whole
//    16-byte chunks, and the permutation is chosen so every 8-lane shared
//    memory phase hits 8 distinct 16-byte bank groups (conflict-free).
//  * Online softmax in the log2 domain with warp-shuffle row max; O is rescaled
//    only when some row's max moved.
//  * merge_kernel (launched behind the decode kernel with programmatic stream
//    serialisation) combines the partials of a segment cut into pieces:
//    M = max_j m_j, out = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kWarps = kDecodeWarpsPerCta;
constexpr int kThreads = kWarps * 32;
constexpr int kBoxBytes = kBlockSize * 128;  // 16 rows x 64 bf16, 128-byte swizzled

template <int D, int NSTAGE>
struct DecodeCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kSlabBytes = kHalves * kBoxBytes;  // one K or V slab of a block
  static constexpr int kStageBytes = 2 * kSlabBytes;
  static constexpr int kRingBytes = NSTAGE * kStageBytes;
  static constexpr int kBarOffset = kWarps * kRingBytes;
  // barriers: the warps' own rings use kWarps * NSTAGE; a shared-prefix CTA uses
  // that many full and as many empty barriers for its pooled ring
  static constexpr int kFlagOffset = kBarOffset + 2 * kWarps * NSTAGE * 8;
  static constexpr int kSmemBytes = kFlagOffset + kWarps * NSTAGE * 4 + 1024;
};

struct DecodeParams {
  const __nv_bfloat16 *q;
  __nv_bfloat16 *out;
  const int32_t *cu_q_lens;
  const int32_t *context_lens;
  const int32_t *block_tables;
  const int32_t *warp_begin;
  const WarpHead *warp_head;
  const Piece *pieces;
  const SharedItem *shared;    // shared-prefix CTAs, after the num_indep_ctas CTAs of warp ranges
  int32_t num_indep_ctas;
  int32_t num_shared_items;    // entries of `shared` (the pairs' chains)
  const MergeGroup *merges;
  float *part_o;
  float2 *part_ml;
  const float *ppart_o;
  const float2 *ppart_ml;
  int32_t *dev_status;
  int32_t lookahead;           // plan sized for this many further steps (chained decode)
  int32_t after_prefill;       // launched right behind this call's tensor-core kernel: the
                               // pool is complete when this kernel starts (that kernel lets
                               // it launch only after its own wait for the append), so no
                               // wait precedes the pool reads; every warp waits at its end
                               // instead, so this kernel completes after that one
  int32_t num_merges;          // all merge groups: decode ones, then prefill ones
  int32_t num_decode_merges;
  int32_t merge_lanes_log2;    // lanes that share one decode row's splits (merge kernel)
  int32_t merge_rows;          // rows the merge launch covers per decode group
  int32_t num_partials;
  int32_t num_warps;
  int32_t num_seqs;
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  float scale_log2;
  int64_t total_q;
  const uint8_t *pool;  // for address-translation warm-up only (data goes through pool_map)
  int64_t pool_bytes;
};

// Byte offset of 16-byte chunk `chunk` (0 .. D/8-1) of key row `row` (0..15) of
// a paged block as one 4-D TMA box lands it: [8-row group][64-column half]
// [8 rows][128 B], 128-byte swizzled (the 16-byte chunk index XOR the row within
// its 8-row atom).
template <int kHalves>
__device__ __forceinline__ uint32_t blk_off(int row, int chunk) {
  return (uint32_t)((((row >> 3) * kHalves + (chunk >> 3)) << 10) + ((row & 7) << 7) +
                    (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D>
__device__ __forceinline__ void write_piece(const DecodeParams &p, const Piece &pc,
                                            float (&o)[D / 8][4], float m_lo, float m_hi,
                                            float l_lo, float l_hi, int R, int cu0, int r, int c);

// LSE merge of results whose keys were cut into several parts (decode segments
// cut into several pieces; prefill sub-tiles cut into several work items):
//   M = max_j m_j,  out = sum_j 2^(m_j - M) O_j / sum_j 2^(m_j - M) l_j.
// One thread per (merge group, row, 4 output columns) makes a single pass over
// the group's splits with a running max (each new split rescales the running
// sums), unrolled so several splits' loads are in flight at once.  A decode row
// with many splits has them dealt out over 2^merge_lanes_log2 adjacent lanes
// (split j to lane j mod that count), whose (M, L, O) are then combined by the
// same rule with xor shuffles, so the loads of all its splits are in flight
// together.  Decode groups come first (partial slots of 16 rows), then prefill
// groups (slots of 128 rows); both write bf16 rows of out.
constexpr int kMergeThreads = 128;

// Combines one row's 4 columns over partial slots 0, step, 2 step, .. < nsplit
// (slot stride `rows`), kBatch splits' loads issued before any is used,
// returning the unnormalised sum with its max M and
// denominator L.  A split whose m is NaN was written by a piece that found its
// plan disagreeing with the device tables: the row is then `poisoned` and must
// not be written.
template <int D, int kBatch>
__device__ __forceinline__ float4 merge_row(const float2 *ml, const float4 *po, int nsplit,
                                            int step, int rows, float &M, float &L,
                                            bool &poisoned) {
  constexpr int kChunks = D / 4;
  M = -INFINITY;
  L = 0.f;
  poisoned = false;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < nsplit; j0 += kBatch * step) {
    float2 v[kBatch];
    float4 x[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {  // predicated: nothing is loaded past the last split
      const int j = j0 + u * step;
      const bool in = j < nsplit;
      v[u] = in ? ml[(int64_t)j * rows] : make_float2(-INFINITY, 0.f);
      x[u] = in ? po[(int64_t)j * rows * kChunks] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      poisoned |= v[u].x != v[u].x;
      // skip padding entries and splits in which this row saw no key
      if (v[u].x == -INFINITY || v[u].x != v[u].x) continue;
      const float mn = fmaxf(M, v[u].x);
      const float a = fast_exp2(M - mn), b = fast_exp2(v[u].x - mn);
      L = L * a + v[u].y * b;
      acc.x = acc.x * a + x[u].x * b;
      acc.y = acc.y * a + x[u].y * b;
      acc.z = acc.z * a + x[u].z * b;
      acc.w = acc.w * a + x[u].w * b;
      M = mn;
    }
  }
  return acc;
}

__device__ __forceinline__ void store_row4(__nv_bfloat16 *dst, float4 acc, float L) {
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2 *>(dst) = pk;
}

// A piece that cannot contribute a result (its plan disagrees with the device
// metadata) writes nothing to out; when it is one part of a merge group, every
// row of its partial slot is marked (m = NaN) so the merge writes none of the
// group's rows either.
__device__ __forceinline__ void poison_piece(const DecodeParams &p, int part, int lane) {
  if (part < 0 || part >= p.num_partials) return;
  if (lane < kRowsPerTile)
    p.part_ml[(int64_t)part * kRowsPerTile + lane] = make_float2(__int_as_float(0x7fc00000), 0.f);
}

template <int D, int kBatch>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const DecodeParams p) {
  constexpr int kChunks = D / 4;  // float4 chunks of a row
  const int64_t t0 = (int64_t)blockIdx.x * kMergeThreads + threadIdx.x;
  // decode groups (their first merge_rows rows, 2^lanes_log2 lanes per row and
  // chunk), then prefill groups
  const int n_dg = p.num_decode_merges;
  const int lanes_log2 = p.merge_lanes_log2;
  const int64_t n_dec = ((int64_t)n_dg * p.merge_rows * kChunks) << lanes_log2;
  const bool dec = t0 < n_dec;
  const int S = dec ? 1 << lanes_log2 : 1;
  const int sub = dec ? (int)(t0 & (S - 1)) : 0;
  const int rows = dec ? kRowsPerTile : kPrefillRows;    // rows of a partial slot
  const int mrows = dec ? p.merge_rows : kPrefillRows;  // rows covered per group
  const int64_t tt = dec ? t0 >> lanes_log2 : t0 - n_dec;
  const int64_t gi = tt / (mrows * kChunks);
  const int rem = (int)(tt % (mrows * kChunks));
  const int row = rem / kChunks, ch = rem % kChunks;
  const bool in = gi < (dec ? n_dg : p.num_merges - p.num_decode_merges);
  // the plan is not written by the kernels before this one: the group is read
  // while they finish; only the partials wait
  MergeGroup g;
  if (in) g = p.merges[dec ? gi : p.num_decode_merges + gi];
  pdl_wait();  // the partials are complete and visible
  // every lane of a row's lane group takes the same exits (they depend on the
  // group, row and chunk only)
  if (!in) return;
  const int G = p.group;
  const int nrows = dec ? g.n_q * G : g.n_q;
  if (row >= nrows || nrows > rows || g.seq < 0 || g.seq >= p.num_seqs || g.nsplit < 1 ||
      g.kind != (dec ? 0 : 1) || g.q_row0 < 0 ||
      g.q_row0 + (dec ? g.n_q : nrows) > p.total_q)
    return;
  const int64_t slot0 = (int64_t)g.part0 + sub;  // this lane's first split
  const float2 *ml = (dec ? p.part_ml : p.ppart_ml) + slot0 * rows + row;
  const float4 *po =
      reinterpret_cast<const float4 *>((dec ? p.part_o : p.ppart_o) + (slot0 * rows + row) * D) +
      ch;
  float M, L;
  bool poisoned;
  float4 acc = merge_row<D, kBatch>(ml, po, g.nsplit - sub, S, rows, M, L, poisoned);
  if (S > 1) {
    // lanes sub and sub ^ o hold disjoint sets of the row's splits: combine
    const unsigned mask = ((1u << S) - 1u) << ((threadIdx.x & 31) & ~(S - 1));
    for (int o = 1; o < S; o <<= 1) {
      const float Mo = __shfl_xor_sync(mask, M, o);
      const float Lo = __shfl_xor_sync(mask, L, o);
      float4 ao;
      ao.x = __shfl_xor_sync(mask, acc.x, o);
      ao.y = __shfl_xor_sync(mask, acc.y, o);
      ao.z = __shfl_xor_sync(mask, acc.z, o);
      ao.w = __shfl_xor_sync(mask, acc.w, o);
      poisoned = __shfl_xor_sync(mask, (int)poisoned, o) != 0 || poisoned;
      const float mn = fmaxf(M, Mo);
      const float a = M == -INFINITY ? 0.f : fast_exp2(M - mn);
      const float b = Mo == -INFINITY ? 0.f : fast_exp2(Mo - mn);
      L = L * a + Lo * b;
      acc.x = acc.x * a + ao.x * b;
      acc.y = acc.y * a + ao.y * b;
      acc.z = acc.z * a + ao.z * b;
      acc.w = acc.w * a + ao.w * b;
      M = mn;
    }
  }
  if (poisoned || sub != 0) return;
  const int64_t tok = g.q_row0 + (dec ? row / G : row);
  const int hq = dec ? g.h * G + row % G : g.h;
  store_row4(p.out + (tok * p.num_q_heads + hq) * D + 4 * ch, acc, L);
}

// Q fragments (A operand) of a row group: rows r and r + 8 of the group's R rows
// (token row / G, head h * G + row % G from packed query row q_row0), head_dim
// permuted to match the K fragments.  Rows >= R read as zeros.
template <int D>
__device__ __forceinline__ void load_q_frags(const DecodeParams &p, int q_row0, int R, int h,
                                             int r, int c, uint32_t (&qa)[D / 16][4]) {
  constexpr int kL = D / 32;
  const int G = p.group;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = r + 8 * half;
    const bool rv = row < R;
    const __nv_bfloat16 *qrow =
        p.q + ((int64_t)(q_row0 + (rv ? row / G : 0)) * p.num_q_heads + h * G +
               (rv ? row % G : 0)) * D;
#pragma unroll
    for (int L = 0; L < kL; ++L) {
      const int e = 8 * (L >> 1) + 2 * c + (L & 1);
      const uint4 v = rv ? ldg128_nc(qrow + 8 * e) : make_uint4(0, 0, 0, 0);
      qa[2 * L][half] = v.x;
      qa[2 * L][2 + half] = v.y;
      qa[2 * L + 1][half] = v.z;
      qa[2 * L + 1][2 + half] = v.w;
    }
  }
}

// One paged block (16 keys at positions p0 ..) of a row group: S = Q K^T, causal
// mask, online softmax in log2 units, O += P V.  sK / sV: the block's K and V in
// shared memory (blk_off layout).  The warp's running (m, l, O) are updated.
template <int D>
__device__ __forceinline__ void block_update(uint32_t sK, uint32_t sV, const uint32_t (&qa)[D / 16][4],
                                             int p0, int q_pos0, int lim_lo, int lim_hi, float sl2,
                                             int r, int c, float &m_lo, float &m_hi, float &l_lo,
                                             float &l_hi, float (&o)[D / 8][4]) {
  constexpr int kL = D / 32;
  constexpr int kNt = D / 8;
  constexpr int kHalves = D / 64;
  // S = Q K^T for the block's 16 keys (two n-tiles of 8 keys)
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    const int t = r + 8 * nt;
#pragma unroll
    for (int L = 0; L < kL; ++L) {
      const int e = 8 * (L >> 1) + 2 * c + (L & 1);
      const uint4 kv = lds128(sK + blk_off<kHalves>(t, e));
      mma_16816(s[nt], qa[2 * L][0], qa[2 * L][1], qa[2 * L][2], qa[2 * L][3], kv.x, kv.y);
      mma_16816(s[nt], qa[2 * L + 1][0], qa[2 * L + 1][1], qa[2 * L + 1][2],
                qa[2 * L + 1][3], kv.z, kv.w);
    }
  }
  // scale to log2 units; causal / context mask on the boundary blocks
  const bool need_mask = p0 + kBlockSize - 1 > q_pos0;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float x = s[nt][j] * sl2;
      if (need_mask) {
        const int pos = p0 + 8 * nt + 2 * c + (j & 1);
        if (pos > (j < 2 ? lim_lo : lim_hi)) x = -INFINITY;
      }
      s[nt][j] = x;
    }
  // online softmax (rows r and r + 8; the 4 lanes of a row hold 4 keys each)
  float mx_lo = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx_hi = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
  mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
  mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
  mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
  const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
  const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
  const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
  const float a_lo = fast_exp2(m_lo - base_lo), a_hi = fast_exp2(m_hi - base_hi);
  m_lo = mn_lo;
  m_hi = mn_hi;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    s[nt][0] = fast_exp2(s[nt][0] - base_lo);
    s[nt][1] = fast_exp2(s[nt][1] - base_lo);
    s[nt][2] = fast_exp2(s[nt][2] - base_hi);
    s[nt][3] = fast_exp2(s[nt][3] - base_hi);
  }
  l_lo = l_lo * a_lo + (s[0][0] + s[0][1]) + (s[1][0] + s[1][1]);
  l_hi = l_hi * a_hi + (s[0][2] + s[0][3]) + (s[1][2] + s[1][3]);
  if (__any_sync(0xffffffffu, a_lo != 1.f || a_hi != 1.f)) {
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt) {
      o[nt][0] *= a_lo;
      o[nt][1] *= a_lo;
      o[nt][2] *= a_hi;
      o[nt][3] *= a_hi;
    }
  }
  // P (bf16) as the A operand: keys are the k dimension
  const uint32_t pa0 = pack_bf16x2(s[0][0], s[0][1]);
  const uint32_t pa1 = pack_bf16x2(s[0][2], s[0][3]);
  const uint32_t pa2 = pack_bf16x2(s[1][0], s[1][1]);
  const uint32_t pa3 = pack_bf16x2(s[1][2], s[1][3]);
  // O += P V: lane (r, c) reads keys 2c, 2c+1, 2c+8, 2c+9 at head_dim chunk r (+8 per half)
#pragma unroll
  for (int hh = 0; hh < kHalves; ++hh) {
    const int ch = hh * 8 + r;  // head_dim chunk
    const uint4 v0 = lds128(sV + blk_off<kHalves>(2 * c, ch));
    const uint4 v1 = lds128(sV + blk_off<kHalves>(2 * c + 1, ch));
    const uint4 v2 = lds128(sV + blk_off<kHalves>(2 * c + 8, ch));
    const uint4 v3 = lds128(sV + blk_off<kHalves>(2 * c + 9, ch));
    const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w};
    const uint32_t w1[4] = {v1.x, v1.y, v1.z, v1.w};
    const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w};
    const uint32_t w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      mma_16816(o[8 * hh + 2 * k], pa0, pa1, pa2, pa3, __byte_perm(w0[k], w1[k], 0x5410),
                __byte_perm(w2[k], w3[k], 0x5410));
      mma_16816(o[8 * hh + 2 * k + 1], pa0, pa1, pa2, pa3,
                __byte_perm(w0[k], w1[k], 0x7632), __byte_perm(w2[k], w3[k], 0x7632));
    }
  }
}

// Shared-block CTA: two independent pairs of warps.  Each pair runs a chain of
// items one after another (its first item at index = pair, then through
// SharedItem::next) -- an item is up to two row groups that read the same
// blocks: the row groups of one verify window wider than 16 rows, or row groups
// of sequences whose tables hold the same prefix blocks -- and streams each
// item's blocks once through a ring pooled from its two warps' rings.  The
// pair's first warp resolves the block tables and issues the copies, running
// ahead across item boundaries; a stage is refilled once both warps have
// released it (an empty mbarrier with two arrivals).  An item with no row group
// contributes nothing; an invalid item is reported and skipped; a `next` that
// is not a later index inside the array ends the chain.  Every wait is bounded.
template <int D, int NSTAGE>
__device__ __forceinline__ void shared_cta(const CUtensorMap &pool_map, const DecodeParams &p,
                                           uint8_t *smem, int warp, int lane) {
  using C = DecodeCfg<D, NSTAGE>;
  constexpr int kS = kSharedRowGroups * NSTAGE;  // stages of a pair's pooled ring
  constexpr int kL = D / 32, kNt = D / 8;
  const int r = lane >> 2, c = lane & 3;
  const int G = p.group, hkv = p.num_kv_heads;
  const int pair = warp / kSharedRowGroups, lw = warp % kSharedRowGroups;
  const int head = (blockIdx.x - p.num_indep_ctas) * kSharedItemsPerCta + pair;
  uint8_t *ring = smem + pair * kSharedRowGroups * C::kRingBytes;  // the pair's warps' rings
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::kBarOffset) + pair * 2 * kS;
  uint64_t *empty = full + kS;
  int *stage_ok = reinterpret_cast<int *>(smem + C::kFlagOffset) + pair * kS;
  if (lw == 0 && lane == 0) {
    for (int s = 0; s < kS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kSharedRowGroups);
    }
    fence_mbar_init();
  }
  auto item_ok = [&](const SharedItem &it) {
    return it.seq0 >= 0 && it.seq0 < p.num_seqs && it.h >= 0 && it.h < hkv && it.kb_begin >= 0 &&
           it.kb_begin <= it.kb_end && it.kb_end <= p.max_blocks_per_seq && it.n_rg >= 1 &&
           it.n_rg <= kSharedRowGroups;
  };
  auto next_of = [&](int idx, const SharedItem &it) {
    return it.next > idx && it.next < p.num_shared_items ? it.next : -1;
  };
  const int first = head < p.num_shared_items ? head : -1;

  // ---- producer state (the pair's first warp; whole warp, uniform): item
  // p_idx, its next block p_j of p_n, and a table window (lane i holds entry
  // win_base + i of the item's sequence)
  int p_idx = first, p_j = 0, p_n = 0, p_seq = 0, p_h = 0, p_kb0 = 0, p_next = -1;
  int win_base = 0, win_val = -1;
  auto p_load = [&](int idx) {
    const SharedItem &it = p.shared[idx];
    const bool ok = item_ok(it);
    p_seq = ok ? it.seq0 : 0;
    p_h = ok ? it.h : 0;
    p_kb0 = ok ? it.kb_begin : 0;
    p_n = ok ? it.kb_end - it.kb_begin : 0;
    p_next = next_of(idx, it);
    p_j = 0;
    win_base = p_kb0;
    win_val = lane < p_n ? __ldg(p.block_tables + (int64_t)p_seq * p.max_blocks_per_seq + p_kb0 + lane)
                         : -1;
  };
  // true when the chain still has a block to issue (moving to later items)
  auto p_more = [&]() {
    while (p_idx >= 0 && p_j >= p_n) {
      p_idx = p_next;
      if (p_idx >= 0) p_load(p_idx);
    }
    return p_idx >= 0;
  };
  if (lw == 0 && first >= 0) p_load(first);

  // ---- the consumers' first item: q rows, lengths and the first table window
  // are not written by the kernels this one follows: read before the wait
  // the current item: the fields used, its checks, this warp's row group
  int c_idx = first, c_h = 0, c_kb0 = 0, c_kb1 = 0, c_next = -1;
  uint32_t qa[2 * kL][4];
  SharedRowGroup rg;
  int cu0 = 0, qs = 0, ctx = 0;
  bool cur_ok = false, has_rg = false, mine = false;
  auto c_setup = [&]() {  // both warps: item c_idx's row group, q and lengths
    const SharedItem &it = p.shared[c_idx];
    cur_ok = item_ok(it);
    const int n_rg = it.n_rg;
    if (!cur_ok && n_rg != 0 && lw == 0 && lane == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
    c_h = cur_ok ? it.h : 0;
    c_kb0 = cur_ok ? it.kb_begin : 0;
    c_kb1 = cur_ok ? it.kb_end : 0;
    c_next = next_of(c_idx, it);
    rg.seq = -1;
    rg.qi0 = rg.n_q = rg.q_row0 = 0;
    rg.part = -1;
    has_rg = cur_ok && lw < n_rg;
    if (has_rg) rg = it.rg[lw];
    mine = has_rg && rg.seq >= 0 && rg.seq < p.num_seqs && rg.qi0 >= 0 &&
           rg.n_q >= 1 && rg.n_q * G <= kRowsPerTile && rg.q_row0 >= 0 &&
           rg.q_row0 + rg.n_q <= p.total_q;
    load_q_frags<D>(p, mine ? rg.q_row0 : 0, mine ? rg.n_q * G : 0, c_h, r, c, qa);
    cu0 = qs = ctx = 0;
    if (mine) {
      cu0 = __ldg(p.cu_q_lens + rg.seq);
      qs = __ldg(p.cu_q_lens + rg.seq + 1) - cu0;
      ctx = __ldg(p.context_lens + rg.seq);
      mine = rg.qi0 + rg.n_q <= qs && qs <= ctx && rg.q_row0 == cu0 + rg.qi0 &&
             c_kb1 <= (ctx + p.lookahead * qs - qs + rg.qi0 + rg.n_q - 1) / kBlockSize + 1;
      if (!mine && lane == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
    }
  };
  if (c_idx >= 0) c_setup();
  __syncthreads();  // barrier initialisation visible to every warp
  if (!p.after_prefill) pdl_wait();

  int issued = 0;  // blocks issued into the pooled ring (the producer's count)
  auto issue = [&]() {  // the pair's first warp, whole warp: the chain's next block
    const int kb = p_kb0 + p_j;
    if (kb >= win_base + 32) {
      win_base = kb;
      win_val = kb + lane < p_kb0 + p_n
                    ? __ldg(p.block_tables + (int64_t)p_seq * p.max_blocks_per_seq + kb + lane)
                    : -1;
    }
    const int phys = __shfl_sync(0xffffffffu, win_val, (kb - win_base) & 31);
    const bool ok = phys >= 0 && phys < p.num_blocks;
    const int s = issued % kS;
    const uint32_t bar = smem_u32(&full[s]);
    if (lane == 0) {
      stage_ok[s] = ok ? 1 : 0;
      if (ok) {
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int row_k = ((phys * 2 + 0) * hkv + p_h) * kBlockSize;
        const uint32_t dst = smem_u32(ring + s * C::kStageBytes);
        tma_load_4d(dst, &pool_map, 0, 0, 0, row_k >> 3, bar);
        tma_load_4d(dst + C::kSlabBytes, &pool_map, 0, 0, 0, (row_k + hkv * kBlockSize) >> 3, bar);
      } else {
        report(p.dev_status, PKV_DEV_BAD_BLOCK);
        mbar_arrive(bar);  // complete the phase without data; the block is skipped
      }
    }
    ++p_j;
    ++issued;
  };
  if (lw == 0)
    for (int k = 0; k < kS && p_more(); ++k) issue();

  const float sl2 = p.scale_log2;
  bool good = true;
  int done = 0;  // blocks consumed (both warps walk the same chain)
  while (c_idx >= 0 && good) {
    const int R = mine ? rg.n_q * G : 0;
    const int q_pos0 = ctx - qs + rg.qi0;
    const int lim_lo = r < R ? q_pos0 + r / G : -1;
    const int lim_hi = r + 8 < R ? q_pos0 + (r + 8) / G : -1;
    const int kb0 = c_kb0;
    const int nblk = c_kb1 - c_kb0;
    float o[kNt][4];
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    for (int j = 0; j < nblk; ++j) {
      const int s = done % kS;
      const uint32_t par = (uint32_t)((done / kS) & 1);
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&full[s]), par))) {
        if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
        good = false;
        break;
      }
      ++done;
      if (mine && stage_ok[s]) {
        const uint32_t sK = smem_u32(ring + s * C::kStageBytes);
        block_update<D>(sK, sK + C::kSlabBytes, qa, (kb0 + j) * kBlockSize, q_pos0, lim_lo,
                        lim_hi, sl2, r, c, m_lo, m_hi, l_lo, l_hi, o);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
      if (lw == 0 && p_more()) {  // refill once both warps released the stage
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[s]), par))) {
          if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
          good = false;
          break;
        }
        issue();
      }
    }
    if (!good) break;
    if (mine) {
      Piece pc;
      pc.seq = rg.seq;
      pc.qi0 = rg.qi0;
      pc.n_q = rg.n_q;
      pc.h = c_h;
      pc.kb_begin = kb0;
      pc.kb_end = c_kb1;
      pc.part = rg.part;
      pc.q_row0 = rg.q_row0;
      write_piece<D>(p, pc, o, m_lo, m_hi, l_lo, l_hi, R, cu0, r, c);
    } else if (has_rg) {  // this warp's row group, which could not be attended
      poison_piece(p, rg.part, lane);
    }
    c_idx = c_next;
    if (c_idx >= 0) c_setup();
  }
  // the issuing warp's copies still in flight land before the CTA exits
  if (lw == 0 && lane == 0)
    for (int j = done; j < issued; ++j)
      mbar_wait(smem_u32(&full[j % kS]), (uint32_t)((j / kS) & 1));
}

template <int D, int NSTAGE>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap pool_map, const DecodeParams p) {
  using C = DecodeCfg<D, NSTAGE>;
  constexpr int kL = D / 32;   // 16-byte Q/K chunks per lane per row
  constexpr int kNt = D / 8;   // n-tiles of the P V product
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  // launched early behind the preceding kernel: let our dependents launch.  The
  // plan, the block tables and q are not written by the kernels this one follows
  // (the KV append writes only the pool), so the warp's range, first piece and
  // sequence lengths are read and its barriers set up before waiting for the
  // predecessor; the pool, the workspace and out are touched only after the wait.
  pdl_trigger();
  if (lane == 0) prefetch_tmap(&pool_map);  // fetched beside the metadata reads below
  if (blockIdx.x >= p.num_indep_ctas) {  // CTA-uniform: a shared-prefix CTA
    shared_cta<D, NSTAGE>(pool_map, p, smem, warp, lane);
    if (p.after_prefill) pdl_wait();
    return;
  }
  const int gw = blockIdx.x * kWarps + warp;
  const bool has_warp = gw < p.num_warps;
  // Start-up is a chain of dependent reads (plan -> pool: the first copies take
  // their block ids from the plan).  After other work has cycled the caches,
  // each step of that chain also pays
  // address-translation misses; touching the pages of the block tables, of the
  // step's small arrays and of the pool now, all independently, takes those
  // misses in parallel with the first read.  (L2 prefetches only: no data is used.)
  {
    constexpr int64_t kPage = 2 << 20;
    const int64_t tab_bytes = (int64_t)p.num_seqs * p.max_blocks_per_seq * 4;
    const int64_t npool = (p.pool_bytes + kPage - 1) / kPage;
    const int nw_all = gridDim.x * kWarps;
    if (lane == 0 && (int64_t)gw * kPage < tab_bytes)
      prefetch_l2(reinterpret_cast<const uint8_t *>(p.block_tables) + (int64_t)gw * kPage);
    if (lane < 4) {  // a few pool pages per warp, spread over the whole pool
      const int64_t pg = (int64_t)gw + (int64_t)lane * nw_all;
      if (pg < npool) prefetch_l2(p.pool + pg * kPage);
    }
    if (gw == 0 && lane == 4) prefetch_l2(p.cu_q_lens);
    if (gw == 0 && lane == 5) prefetch_l2(p.context_lens);
    if (gw == 0 && lane == 6) prefetch_l2(p.q);
  }
  const int pb = has_warp ? __ldg(p.warp_begin + gw) : 0;
  const int pe = has_warp ? __ldg(p.warp_begin + gw + 1) : 0;
  Piece pp;
  int fb0 = -1, fb1 = -1, fb2 = -1;  // physical ids of the first piece's first blocks, if known
  if (has_warp) {
    const WarpHead &wh = p.warp_head[gw];  // pp == pieces[pb], loaded beside the range
    pp = wh.first;
    fb0 = wh.blk[0];
    fb1 = wh.blk[1];
    fb2 = wh.blk[2];
  }
  const int hkv = p.num_kv_heads;
  const int G = p.group;
  int win_base = 0, win_val = -1;  // table window: lane i holds entry win_base + i
  bool win_ok = false;
  // The first copies use the block ids the plan carries, so no table read sits
  // between the plan read and the first copy; lanes 0-2 read the same entries
  // from the device table here, checked once the first block has landed.
  int head_chk = -1;
  if (has_warp && pb < pe && pp.seq >= 0 && pp.seq < p.num_seqs && pp.kb_begin >= 0 &&
      lane < kHeadBlocks && pp.kb_begin + lane < min(pp.kb_end, p.max_blocks_per_seq))
    head_chk = __ldg(p.block_tables + (int64_t)pp.seq * p.max_blocks_per_seq + pp.kb_begin + lane);
  // the first piece's sequence lengths, also ahead of the wait
  int f_cu0 = 0, f_cu1 = 0, f_ctx = 0;
  if (has_warp && pb < pe && pp.seq >= 0 && pp.seq < p.num_seqs) {
    f_cu0 = __ldg(p.cu_q_lens + pp.seq);
    f_cu1 = __ldg(p.cu_q_lens + pp.seq + 1);
    f_ctx = __ldg(p.context_lens + pp.seq);
  }
  uint8_t *ring = smem + warp * C::kRingBytes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kBarOffset) + warp * NSTAGE;
  int *stage_ok = reinterpret_cast<int *>(smem + C::kFlagOffset) + warp * NSTAGE;
  if (lane == 0 && has_warp) {
    for (int s = 0; s < NSTAGE; ++s) mbar_init(smem_u32(&bars[s]), 1);
    fence_mbar_init();
  }
  if (!p.after_prefill) pdl_wait();
  if (!has_warp || pb >= pe) {
    if (p.after_prefill) pdl_wait();
    return;
  }
  __syncwarp();

  // ---- producer: walks the warp's pieces block by block.  Called by the whole
  // warp (uniform control flow); lane 0 issues the copies.  The block table is
  // read 32 entries at a time with one coalesced warp load and the entries are
  // shuffled out, so refilling a stage never waits on a dependent global load.
  const Piece first = pp;  // the producer below moves pp ahead of the consumer
  int ppi = pb, pkb = pp.kb_begin, issued = 0;
  auto load_window = [&]() {  // whole warp: entries pkb .. pkb + 31 of pp's table
    win_base = pkb;
    const int idx = pkb + lane;
    win_val = idx < min(pp.kb_end, p.max_blocks_per_seq)
                  ? __ldg(p.block_tables + (int64_t)pp.seq * p.max_blocks_per_seq + idx)
                  : -1;
    win_ok = true;
  };
  auto issue_next = [&](int stage) {
    while (ppi < pe && pkb >= pp.kb_end) {
      if (++ppi < pe) {
        pp = p.pieces[ppi];
        pkb = pp.kb_begin;
        win_ok = false;
        // the consumer reaches this piece NSTAGE blocks later: bring its q rows
        // (n_q tokens x the group's G heads, G * 2D contiguous bytes per token) into L2
        const int lpt = (G * D * 2 + 127) / 128;  // 128-byte lines per token
        const int t = lane / lpt;
        if (t < pp.n_q && pp.q_row0 >= 0 && pp.q_row0 + pp.n_q <= p.total_q && pp.h >= 0 &&
            pp.h < hkv)
          prefetch_l2(p.q + ((int64_t)(pp.q_row0 + t) * p.num_q_heads + pp.h * G) * D +
                      (lane % lpt) * 64);
      }
    }
    if (ppi >= pe) return;
    const uint32_t bar = smem_u32(&bars[stage]);
    const bool in_table = pp.seq >= 0 && pp.seq < p.num_seqs && pp.h >= 0 && pp.h < hkv &&
                          pkb >= 0 && pkb < p.max_blocks_per_seq;
    // the first copies use the block ids the plan carries; no window is read
    // for them (none is pending, so the shuffle below does not wait either)
    const int inl = ppi == pb && issued < kHeadBlocks
                        ? (issued == 0 ? fb0 : issued == 1 ? fb1 : fb2)
                        : -1;
    if (inl < 0 && in_table && (!win_ok || pkb >= win_base + 32)) load_window();
    const int phys = inl >= 0 ? inl : __shfl_sync(0xffffffffu, win_val, (pkb - win_base) & 31);
    const bool ok = in_table && phys >= 0 && phys < p.num_blocks;
    if (lane == 0) {
      stage_ok[stage] = ok ? 1 : 0;
      if (ok) {
        mbar_arrive_expect_tx(bar, C::kStageBytes);
        const int row_k = ((phys * 2 + 0) * hkv + pp.h) * kBlockSize;
        const int row_v = row_k + hkv * kBlockSize;
        const uint32_t dst = smem_u32(ring + stage * C::kStageBytes);
        // one 4-D box per slab: the whole block of one head (rows / 8 = group coordinate)
        tma_load_4d(dst, &pool_map, 0, 0, 0, row_k >> 3, bar);
        tma_load_4d(dst + C::kSlabBytes, &pool_map, 0, 0, 0, row_v >> 3, bar);
      } else {
        report(p.dev_status, in_table ? PKV_DEV_BAD_BLOCK : PKV_DEV_PLAN_MISMATCH);
        mbar_arrive(bar);  // complete the phase without data; the block is skipped
      }
    }
    ++pkb;
    ++issued;
  };
  for (int s = 0; s < NSTAGE; ++s) issue_next(s);
  // the window for the next copies, read while the first ones are in flight
  if (ppi < pe && pkb < pp.kb_end && pp.seq >= 0 && pp.seq < p.num_seqs && pkb >= 0 &&
      pkb < p.max_blocks_per_seq && (!win_ok || pkb >= win_base + 32))
    load_window();

  const float sl2 = p.scale_log2;
  int stage = 0;
  uint32_t phase = 0;
  int consumed = 0;
  bool abandoned = false;

  for (int pi = pb; pi < pe && !abandoned; ++pi) {
    // the producer runs ahead and usually already holds this piece
    const Piece pc = pi == pb ? first : (pi == ppi ? pp : p.pieces[pi]);
    // ---- piece metadata, checked against the device copies of the step arrays
    bool valid = pc.seq >= 0 && pc.seq < p.num_seqs && pc.h >= 0 && pc.h < hkv &&
                 pc.kb_begin >= 0 && pc.kb_begin <= pc.kb_end &&
                 pc.kb_end <= p.max_blocks_per_seq && pc.n_q >= 1 &&
                 pc.n_q * G <= kRowsPerTile && pc.q_row0 >= 0 &&
                 pc.q_row0 + pc.n_q <= p.total_q;
    // ---- Q fragments (A operand), head_dim permuted to match the K fragments.
    // Rows come straight from the plan's packed index (bounds-checked above), so
    // these loads do not wait for the length loads below; a piece that then
    // fails the check (R = 0) uses none of them.
    uint32_t qa[2 * kL][4];
    load_q_frags<D>(p, pc.q_row0, valid ? pc.n_q * G : 0, pc.h, r, c, qa);
    int cu0 = 0, qs = 0, ctx = 0;
    if (valid) {
      cu0 = pi == pb ? f_cu0 : __ldg(p.cu_q_lens + pc.seq);
      qs = (pi == pb ? f_cu1 : __ldg(p.cu_q_lens + pc.seq + 1)) - cu0;
      ctx = pi == pb ? f_ctx : __ldg(p.context_lens + pc.seq);
      valid = pc.qi0 >= 0 && pc.qi0 + pc.n_q <= qs && qs <= ctx && pc.q_row0 == cu0 + pc.qi0 &&
              pc.kb_end <= (ctx + p.lookahead * qs - qs + pc.qi0 + pc.n_q - 1) / kBlockSize + 1;
    }
    if (!valid && lane == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
    const int R = valid ? pc.n_q * G : 0;
    const int q_pos0 = ctx - qs + pc.qi0;  // causal position of the group's first token
    const int lim_lo = r < R ? q_pos0 + r / G : -1;            // last visible key of row r
    const int lim_hi = r + 8 < R ? q_pos0 + (r + 8) / G : -1;  // ... of row r + 8

    float o[kNt][4];
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    bool head_bad = false;  // the plan's block ids for this piece disagree with the table

    for (int kb = pc.kb_begin; kb < pc.kb_end; ++kb) {
      const bool ok = mbar_wait(smem_u32(&bars[stage]), phase);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) report(p.dev_status, PKV_DEV_TIMEOUT);
        abandoned = true;
        break;
      }
      ++consumed;
      if (consumed == 1) {  // the check entries have landed by now: compare the inline ids
        const int want = lane == 0 ? fb0 : lane == 1 ? fb1 : lane == 2 ? fb2 : -1;
        const bool bad = want >= 0 && want != head_chk;
        if (bad) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
        // blocks loaded from ids the table does not hold: nothing of this
        // piece is used or written
        head_bad = __any_sync(0xffffffffu, bad);
      }
      if (valid && !head_bad && stage_ok[stage]) {
        const uint32_t sK = smem_u32(ring + stage * C::kStageBytes);
        block_update<D>(sK, sK + C::kSlabBytes, qa, kb * kBlockSize, q_pos0, lim_lo, lim_hi, sl2,
                        r, c, m_lo, m_hi, l_lo, l_hi, o);
      }
      __syncwarp();
      issue_next(stage);  // refill this stage with the stream's next block
      if (++stage == NSTAGE) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (abandoned) break;
    if (valid && !head_bad)
      write_piece<D>(p, pc, o, m_lo, m_hi, l_lo, l_hi, R, cu0, r, c);
    else
      poison_piece(p, pc.part, lane);
  }
  if (abandoned) {
    // drain this warp's copies still in flight (bounded) before exiting
    for (int j = consumed; j < issued; ++j)
      mbar_wait(smem_u32(&bars[j % NSTAGE]), (uint32_t)((j / NSTAGE) & 1));
  }
  if (p.after_prefill) pdl_wait();
}

// ---- piece epilogue straight from registers: lane (r, c) holds head_dim
// [64j + 16c, 64j + 16c + 16) of rows r and r + 8.  A whole segment writes the
// normalised bf16 output; a split piece writes its fp32 partial (O, m, l).
template <int D>
__device__ __forceinline__ void write_piece(const DecodeParams &p, const Piece &pc,
                                            float (&o)[D / 8][4], float m_lo, float m_hi,
                                            float l_lo, float l_hi, int R, int cu0, int r, int c) {
  const int G = p.group;
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = r + 8 * half;
    if (row >= R) continue;
    const float l = half ? l_hi : l_lo;
    const float m = half ? m_hi : m_lo;
    const int64_t tok = cu0 + pc.qi0 + row / G;
    const int hq = pc.h * G + row % G;
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
      float v[16];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        v[t] = o[8 * j + t][2 * half];
        v[8 + t] = o[8 * j + t][2 * half + 1];
      }
      if (pc.part < 0) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint4 a, b;
        a.x = pack_bf16x2(v[0] * inv, v[1] * inv);
        a.y = pack_bf16x2(v[2] * inv, v[3] * inv);
        a.z = pack_bf16x2(v[4] * inv, v[5] * inv);
        a.w = pack_bf16x2(v[6] * inv, v[7] * inv);
        b.x = pack_bf16x2(v[8] * inv, v[9] * inv);
        b.y = pack_bf16x2(v[10] * inv, v[11] * inv);
        b.z = pack_bf16x2(v[12] * inv, v[13] * inv);
        b.w = pack_bf16x2(v[14] * inv, v[15] * inv);
        uint4 *dst =
            reinterpret_cast<uint4 *>(p.out + (tok * p.num_q_heads + hq) * D + 64 * j + 16 * c);
        dst[0] = a;
        dst[1] = b;
      } else {
        float4 *dst = reinterpret_cast<float4 *>(
            p.part_o + ((int64_t)pc.part * kRowsPerTile + row) * D + 64 * j + 16 * c);
        dst[0] = make_float4(v[0], v[1], v[2], v[3]);
        dst[1] = make_float4(v[4], v[5], v[6], v[7]);
        dst[2] = make_float4(v[8], v[9], v[10], v[11]);
        dst[3] = make_float4(v[12], v[13], v[14], v[15]);
      }
    }
    if (pc.part >= 0 && c == 0)
      p.part_ml[(int64_t)pc.part * kRowsPerTile + row] = make_float2(m, l);
  }
}

// ------------------------------------------------------------------ host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

DecodeParams make_params(const AttnArgs &a) {
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.cu_q_lens = a.cu_q_lens;
  p.context_lens = a.context_lens;
  p.block_tables = a.block_tables;
  p.warp_begin = a.warp_begin;
  p.warp_head = a.warp_head;
  p.shared = a.shared_items;
  p.num_indep_ctas = (a.num_decode_warps + kWarps - 1) / kWarps;
  p.num_shared_items = a.num_shared_items;
  p.pieces = a.pieces;
  p.merges = a.merge_groups;
  p.part_o = a.part_o;
  p.part_ml = reinterpret_cast<float2 *>(a.part_ml);
  p.num_merges = a.num_merge_groups;
  p.lookahead = a.lookahead;
  p.after_prefill = a.num_prefill_tiles > 0 && a.num_prefill_ctas > 0 ? 1 : 0;
  p.num_decode_merges = a.num_decode_merges;
  p.merge_lanes_log2 = 0;
  p.merge_rows = a.merge_rows;
  p.num_partials = a.num_partials;
  p.ppart_o = a.ppart_o;
  p.ppart_ml = reinterpret_cast<const float2 *>(a.ppart_ml);
  p.dev_status = a.dev_status;
  p.num_warps = a.num_decode_warps;
  p.num_seqs = a.num_seqs;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.desc.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.desc.num_kv_heads;
  p.group = a.num_q_heads / a.desc.num_kv_heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.total_q = a.total_q;
  p.pool = static_cast<const uint8_t *>(a.kv_pool);
  p.pool_bytes = (int64_t)a.desc.num_blocks * 2 * a.desc.num_kv_heads * kBlockSize *
                 a.desc.head_dim * 2;
  return p;
}

template <int D, int NSTAGE>
int launch_decode_t(const AttnArgs &a, const CUtensorMap &map) {
  using C = DecodeCfg<D, NSTAGE>;
  auto kern = decode_kernel<D, NSTAGE>;
  cudaError_t e = prepare_kernel<decode_kernel<D, NSTAGE>>(C::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  const unsigned grid = (unsigned)((a.num_decode_warps + kWarps - 1) / kWarps + a.num_shared_ctas);
  profile_begin(PKV_KERNEL_DECODE, a.stream);
  // programmatic launch only when no profiling event sits between us and our
  // predecessor (an event in between would serialise anyway)
  e = launch_kernel(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, a.stream,
                    !profiling_active(), map, make_params(a));
  profile_end(PKV_KERNEL_DECODE, a.stream);
  return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

}  // namespace

int make_pool_map(void *map_out, const void *pool, const pkv_pool_desc &desc) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap *map = static_cast<CUtensorMap *>(map_out);
  // rows of D bf16 ([num_blocks][2][Hkv][16] rows) seen as (64 columns, 8 rows,
  // D/64 column halves, row groups of 8) with strides (2D, 128, 16D) bytes: a box
  // (64, 8, D/64, 2) is one paged block of one head
  const int d = desc.head_dim, halves = d / 64;
  const int64_t rows = (int64_t)desc.num_blocks * 2 * desc.num_kv_heads * kBlockSize;
  cuuint64_t dims[4] = {64, 8, (cuuint64_t)halves, (cuuint64_t)(rows > 0 ? rows / 8 : 1)};
  cuuint64_t strides[3] = {(cuuint64_t)d * 2, 128, (cuuint64_t)d * 2 * 8};
  cuuint32_t box[4] = {64, 8, (cuuint32_t)halves, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pool), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

int launch_decode(const AttnArgs &a, int *launches) {
  if (a.num_decode_warps <= 0 && a.num_shared_ctas <= 0) return 0;
  CUtensorMap map;
  int e = make_pool_map(&map, a.kv_pool, a.desc);
  if (e) return e;
  e = a.desc.head_dim == 128 ? launch_decode_t<128, 3>(a, map) : launch_decode_t<64, 3>(a, map);
  if (!e) {
    ++*launches;
    count_launches(1);
  }
  return e;
}

int launch_merge(const AttnArgs &a, int *launches) {
  if (a.num_merge_groups <= 0) return 0;
  // lanes per decode row: enough that a group of the average split count has
  // all its splits' loads in one batch of 8 per lane (1, 2, 4 or 8 lanes), as
  // long as the decode threads stay within about one resident wave (many
  // groups already keep every SM busy; more threads would only queue)
  const int64_t chunks = a.desc.head_dim / 4;
  int lanes_log2 = 0;
  if (a.num_decode_merges > 0) {
    const int64_t avg = ((int64_t)a.num_partials + a.num_decode_merges - 1) / a.num_decode_merges;
    const int64_t budget = (int64_t)std::max(device_sm_count(), 1) * 1024;
    const int64_t base = (int64_t)a.num_decode_merges * a.merge_rows * chunks;
    while (lanes_log2 < 3 && avg > (8ll << lanes_log2) && (base << (lanes_log2 + 1)) <= budget)
      ++lanes_log2;
  }
  const int64_t threads =
      (((int64_t)a.num_decode_merges * a.merge_rows * chunks) << lanes_log2) +
      (int64_t)(a.num_merge_groups - a.num_decode_merges) * kPrefillRows * chunks;
  const dim3 grid((unsigned)((threads + kMergeThreads - 1) / kMergeThreads));
  const bool pdl = !profiling_active();
  // 8 splits' loads in flight a lane; a grid larger than one wave of that
  // instance (6 CTAs an SM) takes the one with 6, whose registers let 8 CTAs
  // share an SM (shared_prefix_verify's merge 13.9 -> 11.9 us; a 128-CTA grid
  // does better with the 8)
  const bool wide = (int64_t)grid.x > 6ll * std::max(device_sm_count(), 1);
  auto kern = a.desc.head_dim == 128 ? (wide ? merge_kernel<128, 6> : merge_kernel<128, 8>)
                                     : (wide ? merge_kernel<64, 6> : merge_kernel<64, 8>);
  const cudaError_t pe =
      a.desc.head_dim == 128
          ? (wide ? prepare_kernel<merge_kernel<128, 6>>(0) : prepare_kernel<merge_kernel<128, 8>>(0))
          : (wide ? prepare_kernel<merge_kernel<64, 6>>(0) : prepare_kernel<merge_kernel<64, 8>>(0));
  if (pe != cudaSuccess) return (int)pe;
  DecodeParams mp = make_params(a);
  mp.merge_lanes_log2 = lanes_log2;
  profile_begin(PKV_KERNEL_MERGE, a.stream);
  const cudaError_t le = launch_kernel(kern, grid, dim3(kMergeThreads), 0, a.stream, pdl, mp);
  profile_end(PKV_KERNEL_MERGE, a.stream);
  const int e = le != cudaSuccess ? (int)le : (int)cudaGetLastError();
  if (!e) {
    ++*launches;
    count_launches(1);
  }
  return e;
}

}  // namespace pkv
