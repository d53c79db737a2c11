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
// One CTA = two query sub-tiles (x = 0, 1) of 128 tokens x one query head each,
// whose heads share one KV head: every K/V tile is loaded once for both.
// A sub-tile may instead be gathered: 128 rows (query token x query head, all
// G heads of the KV head) from several sequences whose block tables hold the
// same physical blocks over the item's keys -- a shared prefix, read once per
// 128 rows on the tensor cores instead of once per row group.  Its tokens are
// loaded one 3-D box each (G heads x 64 columns), landing at rows t*G .. in the
// same swizzled layout; no mask applies (the planner keeps only keys every row
// sees), and each row's unnormalised result goes to the split-KV kernel's
// partial slot of its row group, where the merge combines it with the rest of
// that row group's keys.
// Eleven warps with fixed roles:
//   warp 8     TMA producer: both Q sub-tiles (3-D tensor map over
//              [total_q][Hq][D]) and, per 128-key tile, K then V into a ring of
//              K/V slots.  One 4-D TMA box is one paged block of one KV head
//              (16 rows x D, both 64-column halves), issued by lanes 0-7 in
//              parallel; blocks past the context are read out of bounds, i.e.
//              zero-filled without memory traffic.
//   warps 9, 10  one thread each issues the MMAs of sub-tile x = warp - 9:
//                S_x  = Q_x K_j^T        (M=128, N=128 keys, K=D; A and B from smem)
//                O_x += P_x V_j          (M=128, N=D, K=128 keys; A = P from TMEM)
//              and signals completion with tcgen05.commit on mbarriers.  A
//              thread that issues a group of MMAs is held for most of its
//              execution time, so one issuer per sub-tile keeps the tensor pipe
//              fed from two threads.  Warp 9 also allocates 512 TMEM columns.
//   warps 4x .. 4x+3  softmax of sub-tile x: warp w owns TMEM lane quarter
//              w % 4, i.e. query rows 32(w%4) .. +31, one row per thread and all
//              128 keys of a tile.  It reads S_x, masks, takes the row max,
//              computes 2^(scale*s - m) and the row sum, and writes P_x as bf16
//              over the first 64 columns of S_x in TMEM, where the PV MMA reads
//              it.  O_x is rescaled in TMEM only when a row's max grows by more
//              than 2^8 (the softmax is exact for any reference point; the
//              threshold only bounds P <= 2^8).
// The two sub-tiles ping-pong on the tensor pipe: while one sub-tile's softmax
// runs, the other's MMAs do.  S_x(j+1) overwrites P_x(j), so it is issued once
// O_x += P_x(j) V_j has completed.
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
constexpr int kSoftmaxWarpsPerSub = 4;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;  // warps kMmaWarp + x issue the MMAs of sub-tile x
constexpr int kThreads = 352;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kMaxSlots = 8;

enum {
  B_Q_FULL = 0,                  // both Q sub-tiles of an item landed
  B_Q_EMPTY = 1,                 // every S MMA of an item completed (one arrival per issuer)
  B_FULL = 2,                    // + slot: K or V tile landed
  B_EMPTY = B_FULL + kMaxSlots,  // + slot: every MMA reading it completed (one per issuer)
  B_S_FULL = B_EMPTY + kMaxSlots,  // + sub-tile: S_x = Q_x K^T completed
  B_P_FULL = B_S_FULL + 2,       // + sub-tile: P_x written to TMEM (4 warps arrive)
  B_O_DONE = B_P_FULL + 2,       // + sub-tile: O_x += P_x V completed
  B_DRAIN = B_O_DONE + 2,        // + sub-tile: every MMA its issuer issued completed
  B_COUNT = B_DRAIN + 2
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
  static constexpr int kSlots = D == 128 ? 5 : kMaxSlots;
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = 2 * kQBytes;
  static constexpr int kOffBar = kOffRing + kSlots * kSlotBytes;
  static constexpr int kUsed = kOffBar + B_COUNT * 8 + 16;
  // at least 120 KB so a second CTA never shares the SM (and its TMEM)
  static constexpr int kSmemBytes = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
  static_assert(kSlots <= kMaxSlots, "ring too deep");
  static_assert(kUsed + 1024 <= 227 * 1024, "shared memory budget");
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap qg_map,
                   const __grid_constant__ CUtensorMap qr_map,
                   const __grid_constant__ CUtensorMap kv_map, const PrefillParams p) {
  using C = PrefillCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // launched early behind the preceding kernel: let our dependents launch.  The
  // plan, q and the step metadata are not written by the kernels this one
  // follows (the KV append writes only the pool), so barriers, TMEM, the work
  // items and the q tiles go ahead; the producer waits for the predecessor
  // before its first pool read, and no other role reads the pool.
  pdl_trigger();
  // this CTA's bin of work items, run one after another; every barrier keeps
  // counting phases across items (an item that fails its checks is skipped by
  // every role alike and reported by the producer)
  const int it0 = __ldg(p.bin_begin + blockIdx.x), it1 = __ldg(p.bin_begin + blockIdx.x + 1);

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    mbar_init(bar(B_Q_EMPTY), 2);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(bar(B_FULL + s), 1);
      mbar_init(bar(B_EMPTY + s), 2);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(B_S_FULL + x), 1);
      mbar_init(bar(B_P_FULL + x), kSoftmaxWarpsPerSub);
      mbar_init(bar(B_O_DONE + x), 1);
    }
    mbar_init(bar(B_DRAIN + 0), 1);
    mbar_init(bar(B_DRAIN + 1), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::alloc(smem_u32(tmem_slot), kTmemCols);
    tc::relinquish_alloc_permit();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S_x at 128 x; O_x at 256 + D x.  P_x overlays S_x columns 0-63.
  auto t_s = [&](int x) { return tmem + (uint32_t)(x * kKeysPerTile); };
  auto t_o = [&](int x) { return tmem + (uint32_t)(2 * kKeysPerTile + x * D); };

  auto fail = [&]() {
    report(p.dev_status, PKV_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == kProducerWarp) {
    // ======================================================== TMA producer (whole warp)
    if (lane == 0) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&qg_map);
      prefetch_tmap(&qr_map);
      prefetch_tmap(&kv_map);
    }
    // Ring load L (counted over the CTA's items) is K_j (even) or V_j (odd) of
    // the current item, in slot L % kSlots.  Lane b < 8 owns paged block b of
    // every tile: it reads that block's table entry once per tile (a coalesced
    // 32-byte load, issued before the wait for a free slot) and issues the
    // block's K and V boxes itself.  The Q tiles of an item wait until every
    // S MMA of the previous item has read its Q (B_Q_EMPTY).
    const int hkv = p.num_kv_heads;
    int L = 0, nq = 0;  // ring loads and Q loads issued
    bool good = true, waited = false;
    for (int it = it0; it < it1 && good; ++it) {
      const ItemMeta m = load_item(p, it);
      if (!m.ok) {
        if (lane == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
        continue;
      }
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      const int32_t *table = p.block_tables + (int64_t)m.t.seq * p.max_blocks_per_seq;
      const int nblk_ctx = (m.ctx + kBlockSize - 1) / kBlockSize;
      // lane b < 8: the physical id of block b of key tile j (-1: none, zero fill)
      auto tile_block = [&](int j) -> int {
        const int kb = j * kBlocksPerTile + lane;
        return lane < kBlocksPerTile && kb < nblk_ctx && kb < p.max_blocks_per_seq
                   ? __ldg(table + kb)
                   : -1;
      };
      int phys_first = tile_block(m.t.kt0);  // read now: it lands while q is loaded
      if (nq > 0 &&
          !__all_sync(0xffffffffu, mbar_wait(bar(B_Q_EMPTY), (uint32_t)((nq - 1) & 1)))) {
        if (lane == 0) fail();
        break;
      }
      const int nsub = m.t.n_q[1] > 0 ? 2 : 1;
      if (!m.gathered) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_Q_FULL), nsub * C::kQBytes);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (x >= nsub) break;
            const uint32_t sq = smem_u32(smem + C::kOffQ + x * C::kQBytes);
#pragma unroll
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(sq + hh * C::kQHalfBytes, &q_map, hh * 64, m.t.hq[x],
                          m.cu0 + m.t.qi0[x], bar(B_Q_FULL));
          }
        }
        __syncwarp();
      } else {
        // one box per token (its G heads x 64 columns, rows t*G ..); a token
        // index outside q reads as zeros (and is reported), so the byte count
        // the barrier expects holds either way
        // a sub-tile of consecutive tokens is one box of 128 / G tokens (rows
        // past its n_q * G hold other tokens or zeros and are masked); any
        // other gets one box per token
        const int G = p.group, row_bytes = G * 128, run_tokens = kPrefillRows / G;
        const bool r0 = (m.t.runs & 1) != 0, r1 = nsub > 1 && (m.t.runs & 2) != 0;
        const int n0 = m.t.n_q[0], n1 = nsub > 1 ? m.t.n_q[1] : 0;
        const int l0 = r0 ? 0 : n0, l1 = r1 ? 0 : n1;  // tokens loaded one by one
        if (lane == 0) {
          mbar_arrive_expect_tx(
              bar(B_Q_FULL),
              ((r0 ? run_tokens : n0) + (nsub > 1 ? (r1 ? run_tokens : n1) : 0)) * row_bytes *
                  C::kHalves);
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!(x ? r1 : r0)) continue;
            const uint32_t sq = smem_u32(smem + C::kOffQ + x * C::kQBytes);
#pragma unroll
            for (int hh = 0; hh < C::kHalves; ++hh)
              tma_load_3d(sq + hh * C::kQHalfBytes, &qr_map, hh * 64, m.t.h * G,
                          x ? m.t.qi0[1] : m.t.qi0[0], bar(B_Q_FULL));
          }
        }
        __syncwarp();
        // token tk = lane + 32 r of sub-tile x (<= 128 tokens each): all token
        // indices are read first, so their latencies overlap
        int qt[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int x = i >> 2, tk = lane + 32 * (i & 3);
          qt[i] = tk < (x ? l1 : l0) ? __ldg(&p.gather[(x ? m.t.gather[1] : m.t.gather[0]) + tk].q_tok)
                                     : 0;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int x = i >> 2, tk = lane + 32 * (i & 3);
          if (tk >= (x ? l1 : l0)) continue;
          if (qt[i] < 0 || qt[i] >= p.total_q) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
          const uint32_t sq = smem_u32(smem + C::kOffQ + x * C::kQBytes) + tk * row_bytes;
#pragma unroll
          for (int hh = 0; hh < C::kHalves; ++hh)
            tma_load_3d(sq + hh * C::kQHalfBytes, &qg_map, hh * 64, m.t.h * G, qt[i], bar(B_Q_FULL));
        }
        __syncwarp();
      }
      ++nq;
      // the pool is the predecessor's output: wait for it before the first copy
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      int g_k = p.pool_groups;  // this lane's K group coordinate for the current tile
      for (int jl = 0; jl < 2 * m.nkt; ++jl) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          good = false;
          break;
        }
        const int j = m.t.kt0 + (jl >> 1);  // absolute key tile
        if ((jl & 1) == 0) {
          const int phys = jl == 0 ? phys_first : tile_block(j);
          g_k = p.pool_groups;  // out of range: zero fill, no memory traffic
          if (phys >= 0 && phys < p.num_blocks)
            g_k = ((phys * 2 + 0) * hkv + m.t.h) * (kBlockSize / 8);
          else if (phys != -1 || (lane < kBlocksPerTile &&
                                  j * kBlocksPerTile + lane < min(nblk_ctx, p.max_blocks_per_seq)))
            report(p.dev_status, PKV_DEV_BAD_BLOCK);
        }
        const int s = L % C::kSlots;
        if (L >= C::kSlots &&
            !__all_sync(0xffffffffu,
                        mbar_wait(bar(B_EMPTY + s), (uint32_t)(((L / C::kSlots) - 1) & 1)))) {
          if (lane == 0) fail();
          good = false;
          break;
        }
        if (lane == 0) mbar_arrive_expect_tx(bar(B_FULL + s), C::kSlotBytes);
        __syncwarp();
        if (lane < kBlocksPerTile) {
          const int g =
              (jl & 1) == 0 || g_k == p.pool_groups ? g_k : g_k + hkv * (kBlockSize / 8);
          tma_load_4d(smem_u32(smem + C::kOffRing + s * C::kSlotBytes) + lane * C::kBlockBytes,
                      &kv_map, 0, 0, 0, g, bar(B_FULL + s));
        }
        ++L;
      }
    }
    // the kernel must not complete before its predecessor (the next kernel's
    // wait covers ours only), even when this CTA had no valid item
    if (!waited) pdl_wait();
    // our copies still in flight land before the CTA can exit: only the last
    // load of each slot can be pending (a slot is refilled after it was consumed)
    if (lane == 0) {
      for (int l = max(0, L - C::kSlots); l < L; ++l)
        mbar_wait(bar(B_FULL + l % C::kSlots), (uint32_t)((l / C::kSlots) & 1));
      if (nq > 0) mbar_wait(bar(B_Q_FULL), (uint32_t)((nq - 1) & 1));
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ======================================================== MMA issuer of sub-tile x
    // Per item: S_x(0), then per key tile j < nt_x: O_x += P_x(j) V_j, S_x(j+1).
    // While sub-tile x's softmax of tile j runs, its issuer waits and the
    // other sub-tile's MMAs run.  S_x of any tile waits for the previous
    // O_x += P_x V (it writes over P_x), also across items; the first
    // O_x += P_x V of an item needs nothing more, since the softmax warps finish
    // reading O_x of the previous item before they write the new P_x.  Both
    // issuers arrive (tcgen05.commit) on the release of every ring slot and of
    // Q once per use, in ring order, also for key tiles past their own nt_x;
    // each waits for a slot's load before releasing it, so an issuer running
    // ahead never arrives on the slot's next use early.  Waits are bounded
    // (PKV_DEV_TIMEOUT) and stop at an abort.
    if (lane == 0) {
      const int x = warp - kMmaWarp;
      constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kPrefillRows, kKeysPerTile, 0, 0);
      constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kPrefillRows, D, 0, 1);
      auto wait = [&](int b, int parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait(bar(b), (uint32_t)(parity & 1))) return true;
        fail();
        return false;
      };
      const uint32_t sq = smem_u32(smem + C::kOffQ + x * C::kQBytes);
      int L0 = 0, nq = 0;  // ring index of the item's K_0; items (Q loads) done
      int tx = 0;          // key tiles this sub-tile ran in earlier items
      // S_x(j) = Q_x K_j^T once K_j landed and the previous P_x was consumed
      auto issue_s = [&](int j) -> bool {
        const int L = L0 + 2 * j, s = L % C::kSlots;
        if (!wait(B_FULL + s, L / C::kSlots)) return false;
        if (tx + j > 0 && !wait(B_O_DONE + x, tx + j - 1)) return false;
        tc::fence_after_sync();
        const uint32_t sk = smem_u32(smem + C::kOffRing + s * C::kSlotBytes);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t a =
              tc::smem_desc_sw128(sq + (ks >> 2) * C::kQHalfBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t b =
              tc::smem_desc_sw128(sk + (ks >> 2) * 1024 + (ks & 3) * 32, 16, C::kGroupStride);
          tc::mma_bf16(t_s(x), a, b, kIdescS, ks > 0 ? 1u : 0u);
        }
        tc::commit(bar(B_S_FULL + x));
        return true;
      };
      // O_x += P_x(j) V_j once P_x(j) is in TMEM and V_j landed
      auto issue_pv = [&](int j) -> bool {
        const int L = L0 + 2 * j + 1, s = L % C::kSlots;
        if (!wait(B_P_FULL + x, tx + j)) return false;
        if (!wait(B_FULL + s, L / C::kSlots)) return false;
        tc::fence_after_sync();
        const uint32_t sv = smem_u32(smem + C::kOffRing + s * C::kSlotBytes);
#pragma unroll
        for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
          const uint64_t b = tc::smem_desc_sw128(sv + ks * C::kBlockBytes, 1024, C::kGroupStride);
          tc::mma_bf16_ts(t_o(x), t_s(x) + ks * 8, b, kIdescO, (j > 0 || ks > 0) ? 1u : 0u);
        }
        tc::commit(bar(B_O_DONE + x));
        return true;
      };
      // release ring load L (after its landing, so the arrival is for this use)
      auto release = [&](int L) -> bool {
        if (!wait(B_FULL + L % C::kSlots, L / C::kSlots)) return false;
        tc::commit(bar(B_EMPTY + L % C::kSlots));
        return true;
      };
      bool good = true;
      for (int it = it0; it < it1 && good; ++it) {
        const ItemMeta m = load_item(p, it);
        if (!m.ok) continue;
        const int ntx = x ? m.nt[1] : m.nt[0];
        good = wait(B_Q_FULL, nq);
        if (good && ntx > 0) good = issue_s(0);
        if (good && ntx <= 1) tc::commit(bar(B_Q_EMPTY));  // every S of the item issued
        if (good) good = release(L0);                       // K_0
        for (int j = 0; good && j < m.nkt; ++j) {
          if (j < ntx) {
            good = issue_pv(j);
            if (good && j + 1 < ntx) {
              good = issue_s(j + 1);
              if (good && j + 2 == ntx) tc::commit(bar(B_Q_EMPTY));
            }
          }
          if (good) good = release(L0 + 2 * j + 1);                        // V_j
          if (good && j + 1 < m.nkt) good = release(L0 + 2 * j + 2);      // K_{j+1}
        }
        L0 += 2 * m.nkt;
        tx += ntx;
        ++nq;
      }
      // every MMA issued so far completes before TMEM is released
      tc::commit(bar(B_DRAIN + x));
      mbar_wait(bar(B_DRAIN + x), 0);
    }
  } else {
    // ======================================================== softmax (4 warps per sub-tile)
    const int x = warp >> 2;              // sub-tile
    const int quarter = warp & 3;         // TMEM lane quarter
    const int row = quarter * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint32_t ts = t_s(x) + lane_off, to = t_o(x) + lane_off;
    int run0 = 0;  // key tiles this sub-tile ran in earlier items
    bool good = true;
    for (int it = it0; it < it1 && good; ++it) {
      const ItemMeta m = load_item(p, it);
      // per-sub-tile fields by selects (no dynamically indexed local arrays)
      const int n_q = x ? m.t.n_q[1] : m.t.n_q[0];
      const int ntx = x ? m.nt[1] : m.nt[0];
      if (!m.ok || ntx == 0) continue;
      // last visible key of this row (gathered rows see every key of the item)
      const int rows_x = m.gathered ? n_q * p.group : n_q;
      const int lim = row >= rows_x ? -1
                      : m.gathered  ? INT_MAX / 2
                                    : m.ctx - m.qs + (x ? m.t.qi0[1] : m.t.qi0[0]) + row;
      float m_used = -INFINITY, l = 0.f;
      for (int j = 0; j < ntx; ++j) {
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {
          good = false;
          break;
        }
        if (!__all_sync(0xffffffffu,
                        mbar_wait(bar(B_S_FULL + x), (uint32_t)((run0 + j) & 1)))) {
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
        // scores in the log2 domain are sv * mult: a positive scale is applied in
        // the exponent's FMA; a zero or negative one is applied here first
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
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 4; ++c)  // two per instruction, four chains
#pragma unroll
          for (int i = 0; i < 16; ++i)
            m4[i & 3] = max3(m4[i & 3], __uint_as_float(sv[c][2 * i]),
                             __uint_as_float(sv[c][2 * i + 1]));
        const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * mult;
        // lazy rescale of O_x (TMEM) and l when the max grew by more than 2^8 (O_x
        // itself is rescaled below, once the scores are no longer live)
        const bool need = m_used != -INFINITY && mt > m_used + kRescaleLog2;
        const bool any_need = __any_sync(0xffffffffu, need);
        const float alpha = need ? fast_exp2(m_used - mt) : 1.f;
        if (need) {
          l *= alpha;
          m_used = mt;
        }
        if (m_used == -INFINITY) m_used = mt;  // first keys this row sees
        const float nbase = m_used == -INFINITY ? 0.f : -m_used;
        // p = 2^(sv * mult - m): 0 for masked keys (-inf); packed two per column
        // over S_x columns 0-63
        const uint64_t mx2 = f2_pack(mult, mult), nbx2 = f2_pack(nbase, nbase);
        uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k0 = 32 * c + 2 * i;  // key index of the low element
            float p0, p1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[k0 >> 5][k0 & 31]),
                                     __uint_as_float(sv[k0 >> 5][(k0 & 31) + 1])),
                             mx2, nbx2),
                      p0, p1);
            p0 = fast_exp2(p0);
            p1 = fast_exp2(p1);
            acc[i & 1] = f2_add(acc[i & 1], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
          }
          tc::st16(ts + 16 * c, pk);
        }
        {
          float a0, a1, b0, b1;
          f2_unpack(acc[0], a0, a1);
          f2_unpack(acc[1], b0, b1);
          l += (a0 + a1) + (b0 + b1);
        }
        // O_x is idle here: its last update (P_x(j-1) V) completed before S_x(j)
        // was issued, and the next one waits for this tile's P
        if (any_need) {
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
        if (lane == 0) mbar_arrive(bar(B_P_FULL + x));
      }
      if (!good) break;
      // ---- epilogue: O / l.  The next item's first O_x += P_x V waits for this
      // warp's next P_x, which comes after these TMEM reads.
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(bar(B_O_DONE + x), (uint32_t)((run0 + ntx - 1) & 1)))) {
        fail();
        break;
      }
      tc::fence_after_sync();
      int out_row, hq, part;  // re-read rather than kept live through the tile loop
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
      if (part >= 0) {
        // unnormalised O: each lane holds its row's 32-column chunk as 8 pieces
        // of 16 bytes; transposed within groups of 8 lanes, one store covers
        // 4 rows x 128 contiguous bytes rather than 32 rows x 16 bytes
        const int gl = lane & 7, gbase = lane & ~7;
        float *rows8[8];  // destination rows of this lane's group
#pragma unroll
        for (int k = 0; k < 8; ++k)
          rows8[k] = reinterpret_cast<float *>(
              __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(prow), gbase + k));
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tc::ld32(to + 32 * c, ov);
          tc::wait_ld();
          float4 pc[8];
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            pc[v4] = make_float4(__uint_as_float(ov[4 * v4]), __uint_as_float(ov[4 * v4 + 1]),
                                 __uint_as_float(ov[4 * v4 + 2]), __uint_as_float(ov[4 * v4 + 3]));
          transpose8x8(pc, gl);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (rows8[k]) reinterpret_cast<float4 *>(rows8[k] + 32 * c)[gl] = pc[k];
        }
        if (pml) *pml = make_float2(m_used, l);
        tc::fence_before_sync();
        run0 += ntx;
        continue;
      }
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16 *orow = p.out + ((int64_t)out_row * p.num_q_heads + hq) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t ov[32];
        tc::ld32(to + 32 * c, ov);
        tc::wait_ld();
        if (row < n_q) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(ov[8 * v4 + 0]) * inv, __uint_as_float(ov[8 * v4 + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(ov[8 * v4 + 2]) * inv, __uint_as_float(ov[8 * v4 + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(ov[8 * v4 + 4]) * inv, __uint_as_float(ov[8 * v4 + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(ov[8 * v4 + 6]) * inv, __uint_as_float(ov[8 * v4 + 7]) * inv);
            dst[v4] = w;
          }
        }
      }
      tc::fence_before_sync();
      run0 += ntx;
    }
  }

  // ---- teardown: every role has drained its own asynchronous work
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
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

// 3-D view of q: [total_q][Hq][D], box = `tokens` tokens x `heads` heads x 64
// elements (128 x 1 for contiguous sub-tiles, 1 x G for gathered ones).
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
                     const CUtensorMap &qrmap, const CUtensorMap &kvmap) {
  using C = PrefillCfg<D>;
  auto kern = prefill_kernel<D>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
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
                    a.stream, !profiling_active(), qmap, qgmap, qrmap, kvmap, p);
  profile_end(PKV_KERNEL_PREFILL, a.stream);
  return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

}  // namespace

int launch_prefill(const AttnArgs &a, int *launches) {
  if (a.num_prefill_tiles <= 0 || a.num_prefill_ctas <= 0) return 0;
  CUtensorMap qmap, qgmap, qrmap, kvmap;
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
  e = a.desc.head_dim == 128 ? launch_prefill_t<128>(a, qmap, qgmap, qrmap, kvmap)
                             : launch_prefill_t<64>(a, qmap, qgmap, qrmap, kvmap);
  if (!e) {
    ++*launches;
    count_launches(1);
  }
  return e;
}

}  // namespace pkv
