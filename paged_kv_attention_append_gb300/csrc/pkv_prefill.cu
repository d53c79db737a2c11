// Causal varlen prefill over the paged KV pool on the 5th-generation tensor
// cores (tcgen05 + TMEM).
//
// What it computes: the packed attention of the vllm-metal page ("Replacing
// attention, reusing the rest") for chunked-prefill chunks -- query token i of
// a q_len-token chunk at context ctx sees keys 0 .. ctx - q_len + i, keys read
// through the sequence's block table.  The page's M5 "NAX" prefill kernel
// ("Faster prefill on M5") is the prior art for putting this on the tensor
// units; here QK^T and PV are tcgen05 MMAs with fp32 accumulators in TMEM.
//
// A work item holds two query sub-tiles (x = 0, 1) of 128 tokens x one query
// head each, whose heads share one KV head.  A CTA runs an item's sub-tiles one
// after the other as passes; a pass streams the sub-tile's key tiles.
// A sub-tile may instead be gathered: 128 rows (query token x query head, all
// G heads of the KV head) from several sequences whose block tables hold the
// same physical blocks over the item's keys -- a shared prefix, read once per
// 128 rows on the tensor cores instead of once per row group.  Its tokens are
// loaded one 3-D box each (G heads x 64 columns), landing at rows t*G .. in the
// same swizzled layout; no mask applies (the planner keeps only keys every row
// sees), and each row's unnormalised result goes to the split-KV kernel's
// partial slot of its row group, where the merge combines it with the rest of
// that row group's keys.
// Eight warps with fixed roles:
//   warp 4     TMA producer of the pass's Q sub-tile (3-D tensor map over
//              [total_q][Hq][D]) and, per 128-key tile, of K into a ring of K
//              slots;
//   warp 7     TMA producer of V into a ring of V slots.  The two walk the same
//              tiles independently, so neither ring's slot waits hold up the
//              other's copies.  One 4-D TMA box is one paged block of one KV
//              head (16 rows x D, both 64-column halves), issued by lanes 0-7
//              in parallel; blocks past the context are read out of bounds,
//              i.e. zero-filled without memory traffic.  Block-table entries
//              are read 32 at a time (four tiles), one group ahead.
//   warp 5     allocates 512 TMEM columns; one thread issues S(j) = Q K_j^T
//              (M=128, N=128 keys, K=D; A and B from smem) into S buffer j % 3.
//   warp 6     one thread issues O += P(j) V_j (M=128, N=D, K=128 keys; A = P
//              from TMEM, over the first 64 columns of S buffer j % 3).
//   warps 0-3  softmax: warp w owns TMEM lane quarter w, i.e. query rows
//              32w .. 32w+31, one row per thread and all 128 keys of a tile.
//              It reads S(j), masks, computes 2^(scale*s - m) and the row
//              sum, and writes P(j) as bf16 over the first 64 columns of S(j)
//              in TMEM.  The reference m moves only when a row's max grows by
//              more than 2^8 (the softmax is exact for any reference point; the
//              threshold only bounds P <= 2^8), and then O is rescaled in
//              TMEM; so after a pass's first tile the exponentials are taken
//              against the current reference with the row max found in the
//              same sweep, and a tile whose max moved the reference is redone.
// A pass ends with O / l.  For a whole 128-token sub-tile the softmax warps
// write it as bf16 into a V-ring slot that the V producer leaves empty after
// that pass's tiles (the next pass's first V tiles are not needed before this
// output is written), and thread 0 stores it with one bulk tensor store per
// 64-column half; the slot returns to the producer once the copy has read it.
// Shorter
// sub-tiles store their rows directly, and split or gathered ones write fp32
// partials for the merge; neither takes a slot.
// TMEM holds three S buffers and O (3 x 128 + D <= 512 columns), so S(j+1) and
// S(j+2) are computed while the softmax of tile j runs; S(j+3) reuses the
// buffer of S(j) once O += P(j) V_j has read P(j).  Only the softmax and the
// PV chain are serial per tile; the two issuers keep two independent
// accumulators (an S buffer and O) in flight on the tensor pipe.
// Every wait is bounded; a timeout reports PKV_DEV_TIMEOUT, every role drains
// what it issued, and TMEM is always freed.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_tc.cuh"

namespace pkv {

namespace {

constexpr int kKeysPerTile = 128;
constexpr int kBlocksPerTile = kKeysPerTile / kBlockSize;
constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;   // K tiles and the pass's Q
constexpr int kVProducerWarp = 7;  // V tiles
constexpr int kSWarp = 5;   // issues the S MMAs; owns the TMEM allocation
constexpr int kPvWarp = 6;  // issues the PV MMAs
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxSlots = 4;  // per ring (K, V)
constexpr int kTablePrefetchTiles = 32 / kBlocksPerTile;  // tiles per warp-wide table read

enum {
  B_Q_FULL = 0,                  // the pass's Q sub-tile landed
  B_Q_EMPTY = 1,                 // every S MMA of a pass completed (Q may be reloaded)
  B_FULL = 2,                    // + ring * kMaxSlots + slot: K (ring 0) or V (ring 1) tile landed
  B_EMPTY = B_FULL + 2 * kMaxSlots,  // + ring * kMaxSlots + slot: the MMAs reading it completed
  B_S_FULL = B_EMPTY + 2 * kMaxSlots,  // + buffer: S(j) = Q K_j^T completed
  B_P_FULL = B_S_FULL + kSBufs,  // + buffer: P(j) written to TMEM (4 warps arrive)
  B_FREE = B_P_FULL + kSBufs,    // + buffer: O += P(j) V_j completed (buffer reusable)
  B_DRAIN = B_FREE + kSBufs,     // + issuer: every MMA it issued completed
  B_GATE = B_DRAIN + 2,          // the K producer's wait for the preceding kernel returned
  B_STAGED = B_GATE + 1,         // a pass's output is in its staging slot (4 warps arrive)
  B_COUNT = B_STAGED + 1
};

template <int D>
struct PrefillCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalfBytes = kPrefillRows * 128;  // 128 rows x 64 bf16
  static constexpr int kQBytes = kPrefillRows * D * 2;    // one sub-tile
  static constexpr int kSlotBytes = kKeysPerTile * D * 2;  // one K or V tile
  static constexpr int kBlockBytes = kBlockSize * D * 2;   // one paged block of one head
  // inside a slot, paged block b sits at b * kBlockBytes as
  // [8-row group g (2)][64-column half (kHalves)][8 rows][128 B], 128-byte swizzle
  static constexpr int kGroupStride = kHalves * 1024;
  // slots per ring: K_j is refilled once S(j) completed, V_j once O += P(j) V_j
  // did; S runs up to two tiles ahead of the softmax
  static constexpr int kSlots = D == 128 ? 3 : kMaxSlots;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kQBytes;  // K ring, then V ring
  static constexpr int kOffBar = kOffRing + 2 * kSlots * kSlotBytes;
  static constexpr int kUsed = kOffBar + B_COUNT * 8 + 16;
  // at least 120 KB so a second CTA never shares the SM (and its TMEM)
  static constexpr int kSmemBytes = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
  static_assert(kSlots <= kMaxSlots, "ring too deep");
  static_assert(kUsed + 1024 <= 227 * 1024, "shared memory budget");
  static_assert(kSBufs * kKeysPerTile + D <= (int)kTmemCols, "TMEM budget");
};

struct PrefillParams {
  __nv_bfloat16 *out;
  const int32_t *cu_q_lens;
  const int32_t *context_lens;
  const int32_t *block_tables;
  const int32_t *bin_begin;  // work items of CTA b: tiles[bin_begin[b] .. bin_begin[b+1])
  const PrefillTile *tiles;
  float *ppart_o;     // [part][128][D] fp32: unnormalised O of a sub-tile cut along keys
  float2 *ppart_ml;   // [part][128]: (row max in log2 units, row sum) of the same
  const GatherRow *gather;  // tokens of gathered sub-tiles
  float *dpart_o;     // split-KV partial slots [part][16][D]: gathered rows' results
  float2 *dpart_ml;   // [part][16]
  int32_t num_gather;
  int32_t num_dparts;
  int64_t total_q;
  int32_t *dev_status;
  int32_t num_seqs;
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t pool_groups;  // rows of the pool / 8 (out-of-range group coordinate)
  float scale_log2;
};


// 8 x 8 transpose of 16-byte pieces within each group of 8 lanes: lane g of a
// group holds pieces a[0..7] of row g on entry and piece g of rows 0..7 of its
// group on exit.  Three butterfly stages: at stage s a lane swaps, with lane
// g ^ s, the four pieces whose index differs from g in bit s.
__device__ __forceinline__ void transpose8x8(float4 (&a)[8], int g) {
#pragma unroll
  for (int s = 1; s < 8; s <<= 1) {
    const bool hi = (g & s) != 0;
#pragma unroll
    for (int j0 = 0; j0 < 8; ++j0) {
      if (j0 & s) continue;
      const int j1 = j0 | s;
      const float4 send = hi ? a[j0] : a[j1];
      float4 recv;
      recv.x = __shfl_xor_sync(0xffffffffu, send.x, s);
      recv.y = __shfl_xor_sync(0xffffffffu, send.y, s);
      recv.z = __shfl_xor_sync(0xffffffffu, send.z, s);
      recv.w = __shfl_xor_sync(0xffffffffu, send.w, s);
      if (hi)
        a[j0] = recv;
      else
        a[j1] = recv;
    }
  }
}

// One work item's metadata, computed identically by every role (so every role
// skips the same invalid items and agrees on all barrier phases).
struct ItemMeta {
  PrefillTile t;
  int cu0, qs, ctx;
  int nt[2];  // key tiles sub-tile x runs in this item, from t.kt0 (0 when absent)
  int nkt;    // key tiles loaded: t.kt0 .. t.kt1-1
  bool gathered;  // both present sub-tiles are gathered (else both contiguous)
  bool ok;
};

__device__ __forceinline__ ItemMeta load_item(const PrefillParams &p, int it) {
  ItemMeta m;
  m.t = p.tiles[it];
  const PrefillTile &t = m.t;
  m.gathered = t.gather[0] >= 0;
  // rows of a sub-tile: tokens, or tokens x G heads when gathered
  const int rmul = m.gathered ? p.group : 1;
  bool ok = t.seq >= 0 && t.seq < p.num_seqs && t.h >= 0 && t.h < p.num_kv_heads &&
            t.n_q[0] >= 1 && t.n_q[0] * rmul <= kPrefillRows && t.n_q[1] >= 0 &&
            t.n_q[1] * rmul <= kPrefillRows;
#pragma unroll
  for (int x = 0; x < 2; ++x)
    if (t.n_q[x] > 0) {
      if (m.gathered)
        ok = ok && t.gather[x] >= 0 && t.gather[x] + t.n_q[x] <= p.num_gather && t.part[x] >= 0;
      else
        ok = ok && t.gather[x] < 0 && t.hq[x] / p.group == t.h && t.hq[x] >= 0 &&
             t.hq[x] < p.num_q_heads && t.qi0[x] >= 0;
    }
  ok = ok && t.kt0 >= 0 && t.kt0 < t.kt1;
  m.cu0 = m.qs = m.ctx = 0;
  if (ok) {
    m.cu0 = __ldg(p.cu_q_lens + t.seq);
    m.qs = __ldg(p.cu_q_lens + t.seq + 1) - m.cu0;
    m.ctx = __ldg(p.context_lens + t.seq);
    ok = m.qs <= m.ctx;
    if (m.gathered)  // every row of the table's own sequence sees all of the item's keys
      ok = ok && (int64_t)t.kt1 * kKeysPerTile <= (int64_t)m.ctx - m.qs + 1;
    else
#pragma unroll
      for (int x = 0; x < 2; ++x)
        if (t.n_q[x] > 0) ok = ok && t.qi0[x] + t.n_q[x] <= m.qs;
  }
  int seen[2];  // key tiles sub-tile x sees in all
#pragma unroll
  for (int x = 0; x < 2; ++x)
    seen[x] = !ok || t.n_q[x] == 0 ? 0
              : m.gathered         ? t.kt1
                                   : (m.ctx - m.qs + t.qi0[x] + t.n_q[x] - 1) / kKeysPerTile + 1;
  // the item's key range lies inside what sub-tile 0 sees; a present sub-tile
  // runs at least one of its tiles
  ok = ok && t.kt1 <= seen[0] && (t.n_q[1] == 0 || t.kt0 < seen[1]);
#pragma unroll
  for (int x = 0; x < 2; ++x) m.nt[x] = ok && t.n_q[x] > 0 ? min(t.kt1, seen[x]) - t.kt0 : 0;
  m.nkt = ok ? t.kt1 - t.kt0 : 0;
  m.ok = ok;
  return m;
}

// Whether pass x of an item writes its output through a staging slot: a whole
// 128-token sub-tile of contiguous tokens whose keys are not split, in the
// kernel instance built with staging.  Every role evaluates it alike, so all
// agree on the V ring's staging indices.
template <bool kStage>
__device__ __forceinline__ bool stages_output(const ItemMeta &m, int x) {
  const int nq = x ? m.t.n_q[1] : m.t.n_q[0];
  const int part = x ? m.t.part[1] : m.t.part[0];
  return kStage && !m.gathered && part < 0 && nq == kPrefillRows;
}

// kStage: whole sub-tiles leave through a staging slot and bulk tensor stores
// (the instance for steps without gathered sub-tiles); without it every output
// row is stored directly, which keeps the gathered sub-tiles' code as lean as
// before.  Both compute the same result.
template <int D, bool kStage>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap qg_map,
                   const __grid_constant__ CUtensorMap qr_map,
                   const __grid_constant__ CUtensorMap kv_map,
                   const __grid_constant__ CUtensorMap o_map, const PrefillParams p) {
  using C = PrefillCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Launched early behind the preceding kernel.  The plan, q and the step
  // metadata are not written by the kernels this one follows (the KV append
  // writes only the pool), so barriers, TMEM, the work items and the q tiles
  // go ahead; the producers wait for the predecessor before their first pool
  // read, and no other role reads the pool.  Dependents are let launch only
  // after that wait (each warp once the K producer's wait has returned): the
  // split-KV kernel that follows in the same call then runs beside this one on
  // the other SMs, and finds the pool complete without a wait of its own.
  // this CTA's bin of work items, run one after another, each as one pass per
  // present sub-tile; every barrier keeps counting phases across passes (an
  // item that fails its checks is skipped by every role alike and reported by
  // the producer)
  const int it0 = __ldg(p.bin_begin + blockIdx.x), it1 = __ldg(p.bin_begin + blockIdx.x + 1);

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_EMPTY), 1);
    for (int r = 0; r < 2; ++r)
      for (int s = 0; s < C::kSlots; ++s) {
        mbar_init(bar(B_FULL + r * kMaxSlots + s), 1);
        mbar_init(bar(B_EMPTY + r * kMaxSlots + s), 1);
      }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(bar(B_S_FULL + b), 1);
      mbar_init(bar(B_P_FULL + b), kSoftmaxWarps);
      mbar_init(bar(B_FREE + b), 1);
    }
    mbar_init(bar(B_DRAIN + 0), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    mbar_init(bar(B_GATE), 1);
    mbar_init(bar(B_STAGED), kSoftmaxWarps);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kSWarp) {
    tc::alloc(smem_u32(tmem_slot), kTmemCols);
    tc::relinquish_alloc_permit();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S buffer b at 128 b; O at 384.  P(j) overlays columns 0-63 of
  // its S buffer.
  auto t_s = [&](int b) { return tmem + (uint32_t)(b * kKeysPerTile); };
  const uint32_t t_o = tmem + (uint32_t)(kSBufs * kKeysPerTile);

  auto fail = [&]() {
    report(p.dev_status, PKV_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ======================================================== TMA producers (whole warps)
    // Two warps, one per ring (r = 0: K and the pass's Q; r = 1: V), each
    // walking every pass's key tiles on its own, so a K copy never waits for a
    // V slot (released only by O += P V, well behind the S MMAs) nor a V copy
    // for a K slot.  Load n of ring r (counted over the CTA's passes) sits in
    // slot n % kSlots.  Lane b < 8 issues paged block b of every tile; the
    // table entries of four tiles come with one coalesced read by the whole
    // warp, the next four read while the current ones are used.  The Q
    // sub-tile of a pass waits until every S MMA of the previous pass has read
    // its Q (B_Q_EMPTY).  Only the K warp reports bad items and blocks.
    const int r = warp == kVProducerWarp ? 1 : 0;
    if (lane == 0) {
      if (r == 0) {
        prefetch_tmap(&q_map);
        prefetch_tmap(&qg_map);
        prefetch_tmap(&qr_map);
        prefetch_tmap(&o_map);
      }
      prefetch_tmap(&kv_map);
    }
    const int hkv = p.num_kv_heads;
    int nld = 0;    // loads issued into this warp's ring
    int npass = 0;  // passes (Q loads) issued
    bool good = true, waited = false;
    // one tile of KV head h into ring r; lane b < 8 copies paged block `phys`
    // (-1 or out of range: zero fill)
    auto load_tile = [&](int h, int phys) -> bool {
      const int n = nld, s = n % C::kSlots;
      if (n >= C::kSlots &&
          !__all_sync(0xffffffffu, mbar_wait(bar(B_EMPTY + r * kMaxSlots + s),
                                             (uint32_t)(((n / C::kSlots) - 1) & 1)))) {
        if (lane == 0) fail();
        return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar(B_FULL + r * kMaxSlots + s), C::kSlotBytes);
      __syncwarp();
      if (lane < kBlocksPerTile) {
        int g = p.pool_groups;  // out of range: zero fill, no memory traffic
        if (phys >= 0 && phys < p.num_blocks) g = ((phys * 2 + r) * hkv + h) * (kBlockSize / 8);
        tma_load_4d(smem_u32(smem + C::kOffRing + (r * C::kSlots + s) * C::kSlotBytes) +
                        lane * C::kBlockBytes,
                    &kv_map, 0, 0, 0, g, bar(B_FULL + r * kMaxSlots + s));
      }
      ++nld;
      return true;
    };
    for (int it = it0; it < it1 && good; ++it) {
      const ItemMeta m = load_item(p, it);
      if (!m.ok) {
        if (lane == 0 && r == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
        continue;
      }
      const int32_t *table = p.block_tables + (int64_t)m.t.seq * p.max_blocks_per_seq;
      const int nblk_ctx = (m.ctx + kBlockSize - 1) / kBlockSize;
      const int nblk = min(nblk_ctx, p.max_blocks_per_seq);
      // entry of block `lane` of the four tiles from relative tile 4 k on
      // (-1: past the context or the table, zero fill)
      auto read_group = [&](int k) -> int {
        const int kb = (m.t.kt0 + kTablePrefetchTiles * k) * kBlocksPerTile + lane;
        return kb < nblk ? __ldg(table + kb) : -1;
      };
      for (int x = 0; x < 2 && good; ++x) {
        const int ntx = x ? m.nt[1] : m.nt[0];
        if (ntx == 0) continue;
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          good = false;
          break;
        }
        int ent_cur = read_group(0), ent_next = read_group(1);  // land while q is loaded
        if (r == 0 && npass > 0 &&
            !__all_sync(0xffffffffu, mbar_wait(bar(B_Q_EMPTY), (uint32_t)((npass - 1) & 1)))) {
          if (lane == 0) fail();
          good = false;
          break;
        }
        const uint32_t sq = smem_u32(smem + C::kOffQ);
        const int qi0 = x ? m.t.qi0[1] : m.t.qi0[0];
        if (r == 1) {
          // V warp: no Q
        } else if (!m.gathered) {
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q_FULL), C::kQBytes);
#pragma unroll
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(sq + hh * C::kQHalfBytes, &q_map, hh * 64, x ? m.t.hq[1] : m.t.hq[0],
                          m.cu0 + qi0, bar(B_Q_FULL));
          }
          __syncwarp();
        } else {
          // a sub-tile of consecutive tokens is one box of 128 / G tokens (rows
          // past its n_q * G hold other tokens or zeros and are masked); any
          // other gets one box per token (its G heads x 64 columns, rows t*G ..);
          // a token index outside q reads as zeros (and is reported), so the
          // byte count the barrier expects holds either way
          const int G = p.group, row_bytes = G * 128, run_tokens = kPrefillRows / G;
          const bool run = ((m.t.runs >> x) & 1) != 0;
          const int nx = x ? m.t.n_q[1] : m.t.n_q[0];
          const int lx = run ? 0 : nx;  // tokens loaded one by one
          if (lane == 0) {
            mbar_arrive_expect_tx(bar(B_Q_FULL), (run ? run_tokens : nx) * row_bytes * C::kHalves);
            if (run)
#pragma unroll
              for (int hh = 0; hh < C::kHalves; ++hh)
                tma_load_3d(sq + hh * C::kQHalfBytes, &qr_map, hh * 64, m.t.h * G, qi0,
                            bar(B_Q_FULL));
          }
          __syncwarp();
          // token tk = lane + 32 i (<= 128 tokens): all token indices are read
          // first, so their latencies overlap
          const int gbase = x ? m.t.gather[1] : m.t.gather[0];
          int qt[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tk = lane + 32 * i;
            qt[i] = tk < lx ? __ldg(&p.gather[gbase + tk].q_tok) : 0;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int tk = lane + 32 * i;
            if (tk >= lx) continue;
            if (qt[i] < 0 || qt[i] >= p.total_q) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
#pragma unroll
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(sq + tk * row_bytes + hh * C::kQHalfBytes, &qg_map, hh * 64, m.t.h * G,
                          qt[i], bar(B_Q_FULL));
          }
          __syncwarp();
        }
        ++npass;
        // the pool is the predecessor's output: wait for it before the first copy
        if (!waited) {
          pdl_wait();
          waited = true;
          if (r == 0 && lane == 0) mbar_arrive(bar(B_GATE));
          pdl_trigger();
        }
        // the physical block of this lane (< 8) in relative tile j: checked once
        // per tile; ids past the context (-1) are zero-filled
        auto tile_phys = [&](int j) -> int {
          if ((j % kTablePrefetchTiles) == 0 && j > 0) {
            ent_cur = ent_next;
            ent_next = read_group(j / kTablePrefetchTiles + 1);
          }
          const int e = __shfl_sync(0xffffffffu, ent_cur,
                                    (j % kTablePrefetchTiles) * kBlocksPerTile + (lane & 7));
          const int kb = (m.t.kt0 + j) * kBlocksPerTile + lane;
          if (r == 0 && lane < kBlocksPerTile && ((e != -1 && (e < 0 || e >= p.num_blocks)) ||
                                        (e == -1 && kb < nblk)))
            report(p.dev_status, PKV_DEV_BAD_BLOCK);
          return lane < kBlocksPerTile ? e : -1;
        };
        for (int j = 0; good && j < ntx; ++j) {
          if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            good = false;
            break;
          }
          good = load_tile(m.t.h, tile_phys(j));
        }
        // after a pass that stages its output, the V ring's next index holds no
        // tile: it is that output's staging slot.  Its FULL phase completes
        // here, once its previous occupant was released; the softmax warps
        // release it (EMPTY).
        if (good && r == 1 && stages_output<kStage>(m, x)) {
          const int n = nld, s = n % C::kSlots;
          if (n >= C::kSlots &&
              !__all_sync(0xffffffffu, mbar_wait(bar(B_EMPTY + kMaxSlots + s),
                                                 (uint32_t)(((n / C::kSlots) - 1) & 1)))) {
            if (lane == 0) fail();
            good = false;
            break;
          }
          if (lane == 0) mbar_arrive(bar(B_FULL + kMaxSlots + s));
          __syncwarp();
          ++nld;
        }
      }
    }
    // the kernel must not complete before its predecessor (the next kernel's
    // wait covers ours only), even when this CTA had no valid item
    if (!waited) {
      pdl_wait();
      if (r == 0 && lane == 0) mbar_arrive(bar(B_GATE));
      pdl_trigger();
    }
    // our copies still in flight land before the CTA can exit: only the last
    // load of each slot can be pending (a slot is refilled after it was consumed)
    if (lane == 0) {
      for (int l = max(0, nld - C::kSlots); l < nld; ++l)
        mbar_wait(bar(B_FULL + r * kMaxSlots + l % C::kSlots), (uint32_t)((l / C::kSlots) & 1));
      if (r == 0 && npass > 0) mbar_wait(bar(B_Q_FULL), (uint32_t)((npass - 1) & 1));
    }
  } else if (warp == kSWarp || warp == kPvWarp) {
    // dependents may launch once the pool is known complete (bounded wait)
    if (mbar_wait(bar(B_GATE), 0)) pdl_trigger();
    // ======================================================== MMA issuers
    // Tile g (counted over the CTA's passes) uses S buffer g % 3, load g of the
    // K ring and index g + (passes before it) of the V ring, whose index after
    // each pass is that pass's output staging slot.  The S issuer runs S(g) once K_j landed and O += P(g-3) V has completed (it read P(g-3)
    // from the same buffer); the PV issuer runs O += P(g) V_j once P(g) is in
    // TMEM and V_j landed.  Consecutive PV MMAs accumulate into O in issue
    // order; the softmax rescales O only after waiting for the previous PV.
    // Each issuer releases the ring slots it reads (K: S issuer, V: PV issuer)
    // and the S issuer releases Q after the last S of a pass.  Waits are
    // bounded (PKV_DEV_TIMEOUT) and stop at an abort.
    if (lane == 0) {
      const bool is_s = warp == kSWarp;
      constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kPrefillRows, kKeysPerTile, 0, 0);
      constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kPrefillRows, D, 0, 1);
      auto wait = [&](int b, int parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar(b), (uint32_t)(parity & 1))) return true;
        fail();
        return false;
      };
      const uint32_t sq = smem_u32(smem + C::kOffQ);
      int npass = 0, g = 0;  // passes; tiles
      int nst = 0;           // passes that staged their output (V ring indices)
      bool good = true;
      for (int it = it0; it < it1 && good; ++it) {
        const ItemMeta m = load_item(p, it);
        if (!m.ok) continue;
        for (int x = 0; x < 2 && good; ++x) {
          const int ntx = x ? m.nt[1] : m.nt[0];
          if (ntx == 0) continue;
          if (is_s) {
            good = wait(B_Q_FULL, npass);
            for (int j = 0; good && j < ntx; ++j, ++g) {
              const int s = g % C::kSlots, b = g % kSBufs;
              if (!wait(B_FULL + s, g / C::kSlots)) good = false;
              else if (g >= kSBufs && !wait(B_FREE + b, g / kSBufs - 1)) good = false;
              if (!good) break;
              tc::fence_after_sync();
              const uint32_t sk = smem_u32(smem + C::kOffRing + s * C::kSlotBytes);  // K ring
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t a =
                    tc::smem_desc_sw128(sq + (ks >> 2) * C::kQHalfBytes + (ks & 3) * 32, 16, 1024);
                const uint64_t bd =
                    tc::smem_desc_sw128(sk + (ks >> 2) * 1024 + (ks & 3) * 32, 16, C::kGroupStride);
                tc::mma_bf16(t_s(b), a, bd, kIdescS, ks > 0 ? 1u : 0u);
              }
              tc::commit(bar(B_S_FULL + b));
              tc::commit(bar(B_EMPTY + s));  // K_j
            }
            if (good) tc::commit(bar(B_Q_EMPTY));  // every S of the pass issued
          } else {
            for (int j = 0; good && j < ntx; ++j, ++g) {
              // V ring index: a staging index follows each earlier staged pass
              const int vi = g + nst, s = vi % C::kSlots, b = g % kSBufs;
              if (!wait(B_P_FULL + b, g / kSBufs)) good = false;
              else if (!wait(B_FULL + kMaxSlots + s, vi / C::kSlots)) good = false;
              if (!good) break;
              tc::fence_after_sync();
              const uint32_t sv = smem_u32(smem + C::kOffRing + (C::kSlots + s) * C::kSlotBytes);
#pragma unroll
              for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
                const uint64_t bd =
                    tc::smem_desc_sw128(sv + ks * C::kBlockBytes, 1024, C::kGroupStride);
                tc::mma_bf16_ts(t_o, t_s(b) + ks * 8, bd, kIdescO, (j > 0 || ks > 0) ? 1u : 0u);
              }
              tc::commit(bar(B_FREE + b));
              tc::commit(bar(B_EMPTY + kMaxSlots + s));  // V_j
            }
          }
          ++npass;
          if (stages_output<kStage>(m, x)) ++nst;
        }
      }
      // every MMA issued so far completes before TMEM is released
      const int d = is_s ? 0 : 1;
      tc::commit(bar(B_DRAIN + d));
      mbar_wait(bar(B_DRAIN + d), 0);
    }
  } else if (warp < kSoftmaxWarps) {
    // ======================================================== softmax (4 warps)
    // dependents may launch once the pool is known complete (bounded wait)
    if (__all_sync(0xffffffffu, mbar_wait(bar(B_GATE), 0))) pdl_trigger();
    const int quarter = warp;             // TMEM lane quarter
    const int row = quarter * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint32_t to = t_o + lane_off;
    int g = 0;        // tiles of earlier passes
    int nstaged = 0;  // passes whose output went through a staging slot
    bool good = true;
    for (int it = it0; it < it1 && good; ++it) {
      const ItemMeta m = load_item(p, it);
      if (!m.ok) continue;
      for (int x = 0; x < 2 && good; ++x) {
        // per-sub-tile fields by selects (no dynamically indexed local arrays)
        const int n_q = x ? m.t.n_q[1] : m.t.n_q[0];
        const int ntx = x ? m.nt[1] : m.nt[0];
        if (ntx == 0) continue;
        // last visible key of this row (gathered rows see every key of the item)
        const int rows_x = m.gathered ? n_q * p.group : n_q;
        const int lim = row >= rows_x ? -1
                        : m.gathered  ? INT_MAX / 2
                                      : m.ctx - m.qs + (x ? m.t.qi0[1] : m.t.qi0[0]) + row;
        float m_used = -INFINITY, l = 0.f;
        for (int j = 0; j < ntx; ++j, ++g) {
          const int b = g % kSBufs;
          const uint32_t ts = t_s(b) + lane_off;
          if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            good = false;
            break;
          }
          if (!__all_sync(0xffffffffu,
                          mbar_wait(bar(B_S_FULL + b), (uint32_t)((g / kSBufs) & 1)))) {
            fail();
            good = false;
            break;
          }
          tc::fence_after_sync();
          const int rel = lim - (m.t.kt0 + j) * kKeysPerTile;  // keys k <= rel are visible
          uint32_t sv[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) tc::ld32(ts + 32 * c, sv[c]);
          tc::wait_ld();
          // scores in the log2 domain are sv * mult: a positive scale is applied
          // in the exponent's FMA; a zero or negative one is applied here first
          const float mult = sl2 > 0.f ? sl2 : 1.f;
          if (!(sl2 > 0.f)) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i) sv[c][i] = __float_as_uint(__uint_as_float(sv[c][i]) * sl2);
          }
          if (rel < kKeysPerTile - 1) {  // diagonal tile: invisible keys become -inf
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int i = 0; i < 32; ++i) sv[c][i] = 32 * c + i <= rel ? sv[c][i] : 0xff800000u;
          }
          // p = 2^(sv * mult - m): 0 for masked keys (-inf); packed two per
          // column over columns 0-63 of the S buffer, summed into acc.  With
          // track, the row max of the raw scores comes out of the same pass.
          const uint64_t mx2 = f2_pack(mult, mult);
          uint64_t acc[2];
          float m4[4];
          auto exp_pass = [&](float nbase, bool track) {
            const uint64_t nbx2 = f2_pack(nbase, nbase);
            acc[0] = acc[1] = f2_pack(0.f, 0.f);
            m4[0] = m4[1] = m4[2] = m4[3] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t pk[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int k0 = 32 * c + 2 * i;  // key index of the low element
                const float x0 = __uint_as_float(sv[k0 >> 5][k0 & 31]);
                const float x1 = __uint_as_float(sv[k0 >> 5][(k0 & 31) + 1]);
                if (track) m4[i & 3] = max3(m4[i & 3], x0, x1);
                float p0, p1;
                f2_unpack(f2_fma(f2_pack(x0, x1), mx2, nbx2), p0, p1);
                p0 = fast_exp2(p0);
                p1 = fast_exp2(p1);
                acc[i & 1] = f2_add(acc[i & 1], f2_pack(p0, p1));
                pk[i] = pack_bf16x2(p0, p1);
              }
              tc::st16(ts + 16 * c, pk);
            }
          };
          auto ref_of = [](float m) { return m == -INFINITY ? 0.f : -m; };
          // After a pass's first tile the exponentials go first, against the
          // row's current reference m_used, with the row max taken alongside;
          // they stand unless some row's max passed m_used + 2^8 (or a row saw
          // its first keys), and then the tile is redone as below -- so the
          // result is the same either way, and the max is off the critical path.
          float mt;
          bool redo = true;
          if (j > 0) {
            exp_pass(ref_of(m_used), true);
            mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * mult;
            redo = !(mt <= m_used + kRescaleLog2);
          } else {
            m4[0] = m4[1] = m4[2] = m4[3] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)  // two per instruction, four chains
#pragma unroll
              for (int i = 0; i < 16; ++i)
                m4[i & 3] = max3(m4[i & 3], __uint_as_float(sv[c][2 * i]),
                                 __uint_as_float(sv[c][2 * i + 1]));
            mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * mult;
          }
          // lazy rescale of O (TMEM) and l when the max grew by more than 2^8 (O
          // itself is rescaled below, once the scores are no longer live)
          bool any_need = false;
          float alpha = 1.f;
          if (__any_sync(0xffffffffu, redo)) {
            const bool need = m_used != -INFINITY && mt > m_used + kRescaleLog2;
            any_need = __any_sync(0xffffffffu, need);
            alpha = need ? fast_exp2(m_used - mt) : 1.f;
            if (need) {
              l *= alpha;
              m_used = mt;
            }
            if (m_used == -INFINITY) m_used = mt;  // first keys this row sees
            exp_pass(ref_of(m_used), false);
          }
          {
            float a0, a1, b0, b1;
            f2_unpack(acc[0], a0, a1);
            f2_unpack(acc[1], b0, b1);
            l += (a0 + a1) + (b0 + b1);
          }
          if (any_need) {
            // O may be updated by O += P(g-1) V (j > 0 here: the first tile of a
            // pass never rescales); wait for it, then scale O in TMEM
            const int gp = g - 1;
            if (!__all_sync(0xffffffffu, mbar_wait(bar(B_FREE + gp % kSBufs),
                                                   (uint32_t)((gp / kSBufs) & 1)))) {
              fail();
              good = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tc::ld32(to + 32 * c, ov);
              tc::wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
              tc::st32(to + 32 * c, ov);
            }
          }
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_P_FULL + b));
        }
        if (!good) break;
        // ---- epilogue: O / l, once the pass's last O += P V completed.  The
        // next pass's first O += P V (which overwrites O) waits for this warp's
        // next P, which comes after these TMEM reads.  The row's destination is
        // re-read (rather than kept live through the tile loop) while that last
        // O += P V runs.
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        int out_row, hq, part;
        float *prow = nullptr;  // partial destination of this row, if any
        float2 *pml = nullptr;
        {
          const ItemMeta me = load_item(p, it);
          out_row = me.cu0 + (x ? me.t.qi0[1] : me.t.qi0[0]) + row;
          hq = x ? me.t.hq[1] : me.t.hq[0];
          part = x ? me.t.part[1] : me.t.part[0];
          if (me.gathered) {
            // row (t, g): the split-KV partial slot of token t's row group for
            // this key chunk, at the row of head g
            if (row < rows_x) {
              const GatherRow gr = p.gather[(x ? me.t.gather[1] : me.t.gather[0]) + row / p.group];
              const int slot = gr.part0 + part, srow = gr.row0 + row % p.group;
              if (gr.part0 >= 0 && slot < p.num_dparts && srow >= 0 && srow < kRowsPerTile) {
                prow = p.dpart_o + ((int64_t)slot * kRowsPerTile + srow) * D;
                pml = p.dpart_ml + (int64_t)slot * kRowsPerTile + srow;
              } else {
                report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
              }
            }
          } else if (part >= 0 && row < n_q) {
            // keys of this sub-tile are split over several items: unnormalised O
            // and (m, l) to its partial slot, combined by the merge kernel
            prow = p.ppart_o + ((int64_t)part * kPrefillRows + row) * D;
            pml = p.ppart_ml + (int64_t)part * kPrefillRows + row;
          }
          if (me.gathered) part = 0;  // never written out directly
        }
        const int gl = g - 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(B_FREE + gl % kSBufs), (uint32_t)((gl / kSBufs) & 1)))) {
          fail();
          break;
        }
        tc::fence_after_sync();
        // the row's whole O in one round trip
        uint32_t ov[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc::ld32(to + 32 * c, ov[c]);
        tc::wait_ld();
        if (part >= 0) {
          // unnormalised O: each lane holds its row's 32-column chunk as 8 pieces
          // of 16 bytes; transposed within groups of 8 lanes, one store covers
          // 4 rows x 128 contiguous bytes rather than 32 rows x 16 bytes
          const int gl8 = lane & 7, gbase = lane & ~7;
          float *rows8[8];  // destination rows of this lane's group
#pragma unroll
          for (int k = 0; k < 8; ++k)
            rows8[k] = reinterpret_cast<float *>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(prow), gbase + k));
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float4 pc[8];
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              pc[v4] = make_float4(__uint_as_float(ov[c][4 * v4]), __uint_as_float(ov[c][4 * v4 + 1]),
                                   __uint_as_float(ov[c][4 * v4 + 2]), __uint_as_float(ov[c][4 * v4 + 3]));
            transpose8x8(pc, gl8);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              if (rows8[k]) reinterpret_cast<float4 *>(rows8[k] + 32 * c)[gl8] = pc[k];
          }
          if (pml) *pml = make_float2(m_used, l);
          tc::fence_before_sync();
          continue;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        auto pack8 = [&](const uint32_t *o) {
          uint4 w;
          w.x = pack_bf16x2(__uint_as_float(o[0]) * inv, __uint_as_float(o[1]) * inv);
          w.y = pack_bf16x2(__uint_as_float(o[2]) * inv, __uint_as_float(o[3]) * inv);
          w.z = pack_bf16x2(__uint_as_float(o[4]) * inv, __uint_as_float(o[5]) * inv);
          w.w = pack_bf16x2(__uint_as_float(o[6]) * inv, __uint_as_float(o[7]) * inv);
          return w;
        };
        if (stages_output<kStage>(m, x)) {
          // a whole sub-tile: its rows go as bf16 into the staging slot (the V
          // ring's index after this pass's tiles) in the layout of the output
          // tensor map's 128-byte swizzle (16-byte piece c of row r at
          // r * 128 + (c ^ (r & 7)) * 16 of its 64-column half), and thread 0
          // writes them out with one bulk tensor store per half.  The slot's
          // previous occupant was released long before (bounded wait).
          const int vs = g + nstaged, ss = vs % C::kSlots;
          if (vs >= C::kSlots &&
              !__all_sync(0xffffffffu, mbar_wait(bar(B_EMPTY + kMaxSlots + ss),
                                                 (uint32_t)(((vs / C::kSlots) - 1) & 1)))) {
            fail();
            break;
          }
          uint8_t *stage = smem + C::kOffRing + (C::kSlots + ss) * C::kSlotBytes;
#pragma unroll
          for (int hh = 0; hh < C::kHalves; ++hh)
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4 *>(stage + hh * C::kQHalfBytes + row * 128 +
                                         ((c ^ (row & 7)) << 4)) =
                  pack8(&ov[2 * hh + c / 4][8 * (c % 4)]);
          tc::fence_proxy_async_smem();  // visible to the bulk copy
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_STAGED));
          const uint32_t staged_parity = (uint32_t)(nstaged++ & 1);
          if (warp == 0) {
            bool ok = true;
            if (lane == 0) {
              ok = mbar_wait(bar(B_STAGED), staged_parity);
              if (ok) {
#pragma unroll
                for (int hh = 0; hh < C::kHalves; ++hh)
                  tma_store_3d(&o_map, smem_u32(stage + hh * C::kQHalfBytes), hh * 64, hq,
                               out_row);
                bulk_commit();
                // the slot goes back to the V producer once the copy has read
                // it (waiting here keeps this release out of the tile loop)
                bulk_wait_read();
                mbar_arrive(bar(B_EMPTY + kMaxSlots + ss));
              } else {
                fail();
              }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
          }
        } else {
          __nv_bfloat16 *orow = p.out + ((int64_t)out_row * p.num_q_heads + hq) * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            if (row < n_q) {
              uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) dst[v4] = pack8(&ov[c][8 * v4]);
            }
          }
        }
        tc::fence_before_sync();
      }
    }
    // the last staged output has been written before the CTA exits
    if (warp == 0 && lane == 0) bulk_wait();
  }

  // ---- teardown: every role has drained its own asynchronous work
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kSWarp) {
    tc::fence_after_sync();
    tc::dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  void *ptr = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<EncodeTiledFn>(ptr);
}

// 3-D view of q (or of out, which has its shape): [total_q][Hq][D], box =
// `tokens` tokens x `heads` heads x 64 elements (128 x 1 for contiguous
// sub-tiles, 1 x G for gathered ones).
int make_q_map(CUtensorMap *map, const void *q, int64_t total_q, int hq, int d, int heads,
               int tokens) {
  EncodeTiledFn enc = encoder();
  if (!enc) return (int)cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)(total_q > 0 ? total_q : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)heads, (cuuint32_t)tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

template <int D>
int launch_prefill_t(const AttnArgs &a, const CUtensorMap &qmap, const CUtensorMap &qgmap,
                     const CUtensorMap &qrmap, const CUtensorMap &kvmap,
                     const CUtensorMap &omap) {
  using C = PrefillCfg<D>;
  // staging pays on contiguous prefill; the gathered sub-tiles' passes run
  // faster in the instance without it
  const bool stage = a.num_gather_rows == 0;
  auto kern = stage ? prefill_kernel<D, true> : prefill_kernel<D, false>;
  cudaError_t e = stage ? prepare_kernel<prefill_kernel<D, true>>(C::kSmemBytes)
                        : prepare_kernel<prefill_kernel<D, false>>(C::kSmemBytes);
  if (e != cudaSuccess) return (int)e;
  PrefillParams p;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.cu_q_lens = a.cu_q_lens;
  p.context_lens = a.context_lens;
  p.block_tables = a.block_tables;
  p.bin_begin = a.prefill_begin;
  p.tiles = a.prefill_tiles;
  p.ppart_o = a.ppart_o;
  p.ppart_ml = reinterpret_cast<float2 *>(a.ppart_ml);
  p.gather = a.gather_rows;
  p.num_gather = a.num_gather_rows;
  p.dpart_o = a.part_o;
  p.dpart_ml = reinterpret_cast<float2 *>(a.part_ml);
  p.num_dparts = a.num_partials;
  p.total_q = a.total_q;
  p.dev_status = a.dev_status;
  p.num_seqs = a.num_seqs;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.desc.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.desc.num_kv_heads;
  p.group = a.num_q_heads / a.desc.num_kv_heads;
  p.pool_groups = a.desc.num_blocks * 2 * a.desc.num_kv_heads * (kBlockSize / 8);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  profile_begin(PKV_KERNEL_PREFILL, a.stream);
  e = launch_kernel(kern, dim3((unsigned)a.num_prefill_ctas), dim3(kThreads), C::kSmemBytes,
                    a.stream, !profiling_active(), qmap, qgmap, qrmap, kvmap, omap, p);
  profile_end(PKV_KERNEL_PREFILL, a.stream);
  return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

}  // namespace

int launch_prefill(const AttnArgs &a, int *launches) {
  if (a.num_prefill_tiles <= 0 || a.num_prefill_ctas <= 0) return 0;
  CUtensorMap qmap, qgmap, qrmap, kvmap, omap;
  const int group = a.num_q_heads / a.desc.num_kv_heads;
  int e = make_q_map(&qmap, a.q, a.total_q, a.num_q_heads, a.desc.head_dim, 1, kPrefillRows);
  if (e) return e;
  e = make_q_map(&qgmap, a.q, a.total_q, a.num_q_heads, a.desc.head_dim, group, 1);
  if (e) return e;
  e = make_q_map(&qrmap, a.q, a.total_q, a.num_q_heads, a.desc.head_dim, group,
                 kPrefillRows / group);
  if (e) return e;
  e = make_pool_map(&kvmap, a.kv_pool, a.desc);
  if (e) return e;
  // out has q's shape: whole 128-token sub-tiles are stored through this map
  e = make_q_map(&omap, a.out, a.total_q, a.num_q_heads, a.desc.head_dim, 1, kPrefillRows);
  if (e) return e;
  e = a.desc.head_dim == 128 ? launch_prefill_t<128>(a, qmap, qgmap, qrmap, kvmap, omap)
                             : launch_prefill_t<64>(a, qmap, qgmap, qrmap, kvmap, omap);
  if (!e) {
    ++*launches;
    count_launches(1);
  }
  return e;
}

}  // namespace pkv
