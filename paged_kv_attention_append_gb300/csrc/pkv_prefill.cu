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
// One CTA = 128 query tokens x one query head; ten warps with fixed roles:
//   warp 8     TMA producer: the Q tile (3-D tensor map over [total_q][Hq][D])
//              and, per 128-key tile, 8 paged blocks of K and V (2-D pool map,
//              128-byte swizzle) into a 2-stage ring; blocks past the context
//              are read out of bounds, i.e. zero-filled without HBM traffic.
//   warp 9     allocates 512 TMEM columns; one thread issues the MMAs:
//                S[j % 2] = Q K_j^T        (M=128, N=128 keys, K=D; both K-major)
//                O       += P_j V_j        (M=128, N=D, K=128 keys; V MN-major)
//              and signals completion with tcgen05.commit on mbarriers.
//   warps 0-7  softmax: warps w and w + 4 share TMEM lane quarter w % 4 (query
//              rows 32(w%4) .. +31, one row per thread) and split the 128 keys
//              of a tile: warp w < 4 takes keys 0-63, warp w + 4 keys 64-127.
//              Each reads its half of the S row from TMEM, masks, takes a
//              partial row max, exchanges it with its partner through shared
//              memory (named barrier per warp pair), computes 2^(scale*s - m)
//              and its partial row sum, and writes its half of P as bf16 in the
//              swizzled K-major layout the MMA reads.  Two softmax warps per
//              SM sub-partition hide each other's TMEM and barrier latency.  O is rescaled in TMEM only when a
//              row's max grows by more than 2^8 (the softmax is exact for any
//              reference point; the threshold only bounds P <= 2^8).
//   S is double-buffered in TMEM, so the MMA of S_{j+1} overlaps softmax j.
// Every wait is bounded; a timeout reports PKV_DEV_TIMEOUT, every role drains
// what it issued, and TMEM is always freed.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_tc.cuh"

namespace pkv {

namespace {

constexpr int kKeysPerTile = 128;
constexpr int kBlocksPerTile = kKeysPerTile / kBlockSize;
constexpr int kSoftmaxWarps = 8;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kBoxBytesTC = kBlockSize * 128;  // one paged block of one head: 16 rows x 128 B

enum {
  B_Q_FULL = 0,
  B_K_FULL = 1,    // +stage: K tile landed
  B_V_FULL = 3,    // +stage: V tile landed
  B_K_EMPTY = 5,   // +stage: S = Q K^T that read it completed
  B_V_EMPTY = 7,   // +stage: O += P V that read it completed
  B_S_FULL = 9,    // +buffer
  B_S_FREE = 11,   // +buffer
  B_P_FULL = 13,
  B_O_DONE = 14,
  B_DRAIN = 15,
  B_L_READY = 16,  // partial row sums written (one arrive per softmax warp)
  B_COUNT = 17
};

template <int D>
struct PrefillCfg {
  static constexpr int kHalves = D / 64;
  static constexpr int kHalfBytes = kKeysPerTile * 128;  // 128 rows x 64 bf16
  static constexpr int kQBytes = kPrefillRows * D * 2;
  static constexpr int kKBytes = kKeysPerTile * D * 2;
  static constexpr int kStageBytes = 2 * kKBytes;
  static constexpr int kPBytes = kPrefillRows * kKeysPerTile * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffStage = kOffQ + kQBytes;
  static constexpr int kOffP = kOffStage + 2 * kStageBytes;
  static constexpr int kOffBar = kOffP + kPBytes;
  static constexpr int kOffRed = kOffBar + B_COUNT * 8 + 16;  // row max / sum exchange
  static constexpr int kUsed = kOffRed + 2 * 2 * kPrefillRows * 4;
  // at least 120 KB so a second CTA never shares the SM (and its TMEM)
  static constexpr int kSmemBytes = (kUsed + 1024) > 120 * 1024 ? (kUsed + 1024) : 120 * 1024;
};

struct PrefillParams {
  __nv_bfloat16 *out;
  const int32_t *cu_q_lens;
  const int32_t *context_lens;
  const int32_t *block_tables;
  const PrefillTile *tiles;
  int32_t *dev_status;
  int32_t num_seqs;
  int32_t max_blocks_per_seq;
  int32_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t pool_rows;
  float scale_log2;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap q_map,
                   const __grid_constant__ CUtensorMap pool_map, const PrefillParams p) {
  using C = PrefillCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // launched early behind the preceding kernel: let our dependents launch, then
  // wait for the predecessor's writes (pool, q, metadata) before reading anything
  pdl_trigger();
  pdl_wait();
  const PrefillTile tile = p.tiles[blockIdx.x];

  // ---- tile metadata from the device copies of the step arrays (CTA-uniform)
  bool ok = tile.seq >= 0 && tile.seq < p.num_seqs && tile.hq >= 0 &&
            tile.hq < p.num_q_heads && tile.n_q >= 1 && tile.n_q <= kPrefillRows && tile.qi0 >= 0;
  int cu0 = 0, qs = 0, ctx = 0;
  if (ok) {
    cu0 = __ldg(p.cu_q_lens + tile.seq);
    qs = __ldg(p.cu_q_lens + tile.seq + 1) - cu0;
    ctx = __ldg(p.context_lens + tile.seq);
    ok = tile.qi0 + tile.n_q <= qs && qs <= ctx;
  }
  if (!ok) {
    if (threadIdx.x == 0) report(p.dev_status, PKV_DEV_PLAN_MISMATCH);
    return;
  }
  const int h = tile.hq / p.group;
  const int q_pos0 = ctx - qs + tile.qi0;          // causal position of row 0
  const int ntiles = (q_pos0 + tile.n_q - 1) / kKeysPerTile + 1;
  const int nblk_ctx = (ctx + kBlockSize - 1) / kBlockSize;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B_COUNT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto bar = [&](int i) { return smem_u32(&bars[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar(B_Q_FULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(B_K_FULL + s), 1);
      mbar_init(bar(B_V_FULL + s), 1);
      mbar_init(bar(B_K_EMPTY + s), 1);
      mbar_init(bar(B_V_EMPTY + s), 1);
      mbar_init(bar(B_S_FULL + s), 1);
      mbar_init(bar(B_S_FREE + s), kSoftmaxWarps);
    }
    mbar_init(bar(B_P_FULL), kSoftmaxWarps);
    mbar_init(bar(B_O_DONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    mbar_init(bar(B_L_READY), kSoftmaxWarps);
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
  const uint32_t t_s0 = tmem, t_o = tmem + 2 * kKeysPerTile;

  auto fail = [&]() {
    report(p.dev_status, PKV_DEV_TIMEOUT);
    *abort_flag = 1;
  };

  if (warp == kProducerWarp) {
    // ======================================================== TMA producer (whole warp)
    // Lane b < 8 owns paged block b of every 128-key tile: it reads that block's
    // table entry (one coalesced 32-byte load for the tile, issued before the
    // wait for a free stage so the latency hides behind it) and issues the
    // block's K and V boxes itself.
    if (lane == 0) {
      prefetch_tmap(&q_map);
      prefetch_tmap(&pool_map);
      const uint32_t sq = smem_u32(smem + C::kOffQ);
      mbar_arrive_expect_tx(bar(B_Q_FULL), C::kQBytes);
#pragma unroll
      for (int hh = 0; hh < C::kHalves; ++hh)
        tma_load_3d(sq + hh * C::kHalfBytes, &q_map, hh * 64, tile.hq, cu0 + tile.qi0,
                    bar(B_Q_FULL));
    }
    // K and V of a tile have separate slots: the K slot frees as soon as the
    // S MMA that reads it completes, so K_{j} is loaded one step earlier than
    // V_{j}, which waits for the P V MMA of tile j-2.  Order: K_j, then V_{j-1}.
    const int32_t *table = p.block_tables + (int64_t)tile.seq * p.max_blocks_per_seq;
    const int hkv = p.num_kv_heads;
    int k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
    int prev_row_v = p.pool_rows;
    auto load = [&](int full, int empty, int t, uint32_t dst, int row) -> bool {
      const int s = t & 1;
      if (t >= 2 && !__all_sync(0xffffffffu, mbar_wait(bar(empty + s),
                                                        (uint32_t)(((t >> 1) - 1) & 1)))) {
        if (lane == 0) fail();
        return false;
      }
      if (lane == 0) mbar_arrive_expect_tx(bar(full + s), C::kKBytes);
      __syncwarp();
      if (lane < kBlocksPerTile) {
#pragma unroll
        for (int hh = 0; hh < C::kHalves; ++hh)
          tma_load_2d(dst + hh * C::kHalfBytes + lane * kBoxBytesTC, &pool_map, hh * 64, row,
                      bar(full + s));
      }
      return true;
    };
    bool good = true;
    for (int j = 0; j <= ntiles && good; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
      int row_v = p.pool_rows;
      if (j < ntiles) {
        const int kb = j * kBlocksPerTile + lane;
        int row_k = p.pool_rows;  // out of range: zero fill, no memory traffic
        if (lane < kBlocksPerTile && kb < nblk_ctx && kb < p.max_blocks_per_seq) {
          const int phys = __ldg(table + kb);
          if (phys >= 0 && phys < p.num_blocks) {
            row_k = ((phys * 2 + 0) * hkv + h) * kBlockSize;
            row_v = row_k + hkv * kBlockSize;
          } else {
            report(p.dev_status, PKV_DEV_BAD_BLOCK);
          }
        }
        const uint32_t sk = smem_u32(smem + C::kOffStage + (j & 1) * C::kStageBytes);
        good = load(B_K_FULL, B_K_EMPTY, j, sk, row_k);
        if (!good) break;
        ++k_issued[j & 1];
      }
      if (j >= 1) {
        const int t = j - 1;
        const uint32_t sv = smem_u32(smem + C::kOffStage + (t & 1) * C::kStageBytes) + C::kKBytes;
        good = load(B_V_FULL, B_V_EMPTY, t, sv, prev_row_v);
        if (!good) break;
        ++v_issued[t & 1];
      }
      prev_row_v = row_v;
    }
    // our copies still in flight land before the CTA can exit
    if (lane == 0) {
      for (int s = 0; s < 2; ++s) {
        if (k_issued[s]) mbar_wait(bar(B_K_FULL + s), (uint32_t)((k_issued[s] - 1) & 1));
        if (v_issued[s]) mbar_wait(bar(B_V_FULL + s), (uint32_t)((v_issued[s] - 1) & 1));
      }
      mbar_wait(bar(B_Q_FULL), 0);
    }
  } else if (warp == kMmaWarp) {
    // ======================================================== MMA issuer
    // A non-blocking loop: issue S_ns = Q K_ns^T as soon as K_ns has landed and
    // its S buffer is free, and O += P_npv V_npv as soon as P_npv is written and
    // V_npv has landed -- whichever is ready first, so neither waits behind the
    // other's loads.  Gives up (PKV_DEV_TIMEOUT) after kWaitLimitNs without progress.
    if (lane == 0) {
      constexpr uint32_t kIdescS = tc::idesc_bf16_f32(kPrefillRows, kKeysPerTile, 0, 0);
      constexpr uint32_t kIdescO = tc::idesc_bf16_f32(kPrefillRows, D, 0, 1);
      const uint32_t sq = smem_u32(smem + C::kOffQ);
      const uint32_t sp = smem_u32(smem + C::kOffP);
      bool good = mbar_wait(bar(B_Q_FULL), 0);
      if (!good) fail();
      int ns = 0, npv = 0;
      uint64_t t_last = global_timer_ns();
      while (good && npv < ntiles) {
        bool progressed = false;
        if (ns < ntiles && mbar_test_wait(bar(B_K_FULL + (ns & 1)), (uint32_t)((ns >> 1) & 1)) &&
            (ns < 2 || mbar_test_wait(bar(B_S_FREE + (ns & 1)), (uint32_t)(((ns >> 1) - 1) & 1)))) {
          tc::fence_after_sync();
          const uint32_t sk = smem_u32(smem + C::kOffStage + (ns & 1) * C::kStageBytes);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) {
            const uint64_t a = tc::smem_desc_sw128(
                sq + (ks >> 2) * C::kHalfBytes + (ks & 3) * 32, 16, 1024);
            const uint64_t b = tc::smem_desc_sw128(
                sk + (ks >> 2) * C::kHalfBytes + (ks & 3) * 32, 16, 1024);
            tc::mma_bf16(t_s0 + (ns & 1) * kKeysPerTile, a, b, kIdescS, ks > 0 ? 1u : 0u);
          }
          tc::commit(bar(B_S_FULL + (ns & 1)));
          tc::commit(bar(B_K_EMPTY + (ns & 1)));
          ++ns;
          progressed = true;
        }
        if (npv < ns && mbar_test_wait(bar(B_P_FULL), (uint32_t)(npv & 1)) &&
            mbar_test_wait(bar(B_V_FULL + (npv & 1)), (uint32_t)((npv >> 1) & 1))) {
          tc::fence_after_sync();
          const uint32_t sv =
              smem_u32(smem + C::kOffStage + (npv & 1) * C::kStageBytes) + C::kKBytes;
#pragma unroll
          for (int ks = 0; ks < kKeysPerTile / 16; ++ks) {
            const uint64_t a = tc::smem_desc_sw128(
                sp + (ks >> 2) * C::kHalfBytes + (ks & 3) * 32, 16, 1024);
            const uint64_t b = tc::smem_desc_sw128(sv + ks * 2048, C::kHalfBytes, 1024);
            tc::mma_bf16(t_o, a, b, kIdescO, (npv > 0 || ks > 0) ? 1u : 0u);
          }
          tc::commit(bar(B_O_DONE));
          tc::commit(bar(B_V_EMPTY + (npv & 1)));
          ++npv;
          progressed = true;
        }
        if (progressed) {
          t_last = global_timer_ns();
        } else if (*abort_flag) {
          good = false;
        } else if (global_timer_ns() - t_last > kWaitLimitNs) {
          fail();
          good = false;
        }
      }
      // every MMA issued so far completes before TMEM is released
      tc::commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0);
    }
  } else {
    // ======================================================== softmax (8 warps)
    const int quarter = warp & 3;         // TMEM lane quarter
    const int half = warp >> 2;           // 0: keys 0-63 / O columns [0, D/2); 1: the rest
    const int row = quarter * 32 + lane;  // query row = TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int lim = row < tile.n_q ? q_pos0 + row : -1;  // last visible key of this row
    const float sl2 = p.scale_log2;
    constexpr int kHalfKeys = kKeysPerTile / 2;
    constexpr int kOCols = D / 2;  // O columns owned by this thread
    float m_used = -INFINITY, l = 0.f;  // l: partial row sum over this thread's keys
    bool good = true;
    const uint32_t sp = smem_u32(smem + C::kOffP) + half * C::kHalfBytes;
    float *red = reinterpret_cast<float *>(smem + C::kOffRed);
    for (int j = 0; j < ntiles; ++j) {
      if (__any_sync(0xffffffffu, *abort_flag != 0)) {
        good = false;
        break;
      }
      const int s = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_S_FULL + s), (uint32_t)((j >> 1) & 1)))) {
        fail();
        good = false;
        break;
      }
      tc::fence_after_sync();
      // Both warps of the pair read the whole S row for the row max (no exchange
      // needed: they reach the same max); each keeps only its own 64 keys.
      const int rel = lim - j * kKeysPerTile;  // keys k <= rel are visible
      const bool diag = rel < kKeysPerTile - 1;
      const uint32_t s_base = tmem + lane_off + s * kKeysPerTile;
      float x[kHalfKeys];  // raw scores of this thread's keys
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      const bool fast = sl2 > 0.f && !diag;  // positive scale, every key of the tile visible
      {
        uint32_t mine[2][32], other[2][32];
        tc::ld32(s_base + half * kHalfKeys, mine[0]);
        tc::ld32(s_base + half * kHalfKeys + 32, mine[1]);
        tc::ld32(s_base + (1 - half) * kHalfKeys, other[0]);
        tc::ld32(s_base + (1 - half) * kHalfKeys + 32, other[1]);
        tc::wait_ld();
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
          for (int i = 0; i < 32; ++i) x[32 * k + i] = __uint_as_float(mine[k][i]);
        if (fast) {  // max of the raw scores, two per instruction, four chains
#pragma unroll
          for (int i = 0; i < kHalfKeys / 2; ++i)
            m4[i & 3] = max3(m4[i & 3], x[2 * i], x[2 * i + 1]);
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              m4[i & 3] = max3(m4[i & 3], __uint_as_float(other[k][2 * i]),
                               __uint_as_float(other[k][2 * i + 1]));
        } else {  // diagonal tile or non-positive scale: scaled, masked scores
          const int kb_mine = half * kHalfKeys, kb_other = (1 - half) * kHalfKeys;
#pragma unroll
          for (int i = 0; i < kHalfKeys; ++i)
            m4[i & 3] = fmaxf(m4[i & 3], kb_mine + i <= rel ? x[i] * sl2 : -INFINITY);
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              m4[i & 3] = fmaxf(m4[i & 3], kb_other + 32 * k + i <= rel
                                               ? __uint_as_float(other[k][i]) * sl2
                                               : -INFINITY);
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_FREE + s));
      float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      if (fast) mt *= sl2;
      // lazy rescale of O (TMEM) and l when the max grew by more than 2^8; the two
      // threads of a row take the same decision (same row max)
      const bool need = m_used != -INFINITY && mt > m_used + kRescaleLog2;
      bool o_ready = false;
      if (__any_sync(0xffffffffu, need)) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE), (uint32_t)((j - 1) & 1)))) {
          fail();
          good = false;
          break;
        }
        o_ready = true;
        tc::fence_after_sync();
        const float alpha = need ? fast_exp2(m_used - mt) : 1.f;
#pragma unroll
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t ov[32];
          const uint32_t ta = t_o + lane_off + half * kOCols + 32 * c;
          tc::ld32(ta, ov);
          tc::wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tc::st32(ta, ov);
        }
        tc::wait_st();
        l *= alpha;
        if (need) m_used = mt;
      }
      if (m_used == -INFINITY) m_used = mt;  // first keys this row sees
      const float nbase = m_used == -INFINITY ? 0.f : -m_used;
      // p = 2^(scale_log2 * s - m) for visible keys, 0 for masked ones
      uint32_t pk[kHalfKeys / 2];
      const int rel_mine = rel - half * kHalfKeys;
      const uint64_t sl2x2 = f2_pack(sl2, sl2), nbx2 = f2_pack(nbase, nbase);
      uint64_t acc[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < kHalfKeys / 2; ++i) {
        float p0, p1;
        f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), sl2x2, nbx2), p0, p1);
        p0 = fast_exp2(p0);
        p1 = fast_exp2(p1);
        if (diag) {
          p0 = 2 * i <= rel_mine ? p0 : 0.f;
          p1 = 2 * i + 1 <= rel_mine ? p1 : 0.f;
        }
        acc[i & 1] = f2_add(acc[i & 1], f2_pack(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      {
        float a0, a1, b0, b1;
        f2_unpack(acc[0], a0, a1);
        f2_unpack(acc[1], b0, b1);
        l += (a0 + a1) + (b0 + b1);
      }
      // the P buffer is free once P_{j-1} V_{j-1} completed
      if (j >= 1 && !o_ready) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE), (uint32_t)((j - 1) & 1)))) {
          fail();
          good = false;
          break;
        }
      }
      // this thread's 64 keys = one 128-byte swizzled row of the P half tile
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint32_t addr = sp + row * 128 + ((c ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_FULL));
    }
    // ---- epilogue: the two partial row sums meet in shared memory (every
    // softmax warp arrives exactly once, also after an abort), then O / l
    red[half * kPrefillRows + row] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(B_L_READY));
    const bool l_ok = __all_sync(0xffffffffu, mbar_wait(bar(B_L_READY), 0));
    if (!l_ok) fail();
    if (good && l_ok && !__any_sync(0xffffffffu, *abort_flag != 0)) {
      if (!__all_sync(0xffffffffu, mbar_wait(bar(B_O_DONE), (uint32_t)((ntiles - 1) & 1)))) {
        fail();
      } else {
        tc::fence_after_sync();
        const float lt = red[row] + red[kPrefillRows + row];
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        __nv_bfloat16 *orow =
            p.out + ((int64_t)(cu0 + tile.qi0 + row) * p.num_q_heads + tile.hq) * D + half * kOCols;
#pragma unroll
        for (int c = 0; c < kOCols / 32; ++c) {
          uint32_t ov[32];
          tc::ld32(t_o + lane_off + half * kOCols + 32 * c, ov);
          tc::wait_ld();
          if (row < tile.n_q) {
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
      }
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

// 3-D view of q: [total_q][Hq][D], box = 128 tokens x 1 head x 64 elements.
int make_q_map(CUtensorMap *map, const void *q, int64_t total_q, int hq, int d) {
  typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  void *ptr = nullptr;
  cudaDriverEntryPointQueryResult qr;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                       &qr) != cudaSuccess ||
      qr != cudaDriverEntryPointSuccess)
    return (int)cudaErrorNotSupported;
  EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(ptr);
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hq, (cuuint64_t)(total_q > 0 ? total_q : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hq * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kPrefillRows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

template <int D>
int launch_prefill_t(const AttnArgs &a, const CUtensorMap &qmap, const CUtensorMap &pmap) {
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
  p.tiles = a.prefill_tiles;
  p.dev_status = a.dev_status;
  p.num_seqs = a.num_seqs;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_blocks = a.desc.num_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.desc.num_kv_heads;
  p.group = a.num_q_heads / a.desc.num_kv_heads;
  p.pool_rows = a.desc.num_blocks * 2 * a.desc.num_kv_heads * kBlockSize;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  profile_begin(PKV_KERNEL_PREFILL, a.stream);
  e = launch_kernel(kern, dim3((unsigned)a.num_prefill_tiles), dim3(kThreads), C::kSmemBytes,
                    a.stream, !profiling_active(), qmap, pmap, p);
  profile_end(PKV_KERNEL_PREFILL, a.stream);
  return e != cudaSuccess ? (int)e : (int)cudaGetLastError();
}

}  // namespace

int launch_prefill(const AttnArgs &a, int *launches) {
  if (a.num_prefill_tiles <= 0) return 0;
  CUtensorMap qmap, pmap;
  int e = make_q_map(&qmap, a.q, a.total_q, a.num_q_heads, a.desc.head_dim);
  if (e) return e;
  e = make_pool_map(&pmap, a.kv_pool, a.desc);
  if (e) return e;
  e = a.desc.head_dim == 128 ? launch_prefill_t<128>(a, qmap, pmap)
                             : launch_prefill_t<64>(a, qmap, pmap);
  if (!e) {
    ++*launches;
    count_launches(1);
  }
  return e;
}

}  // namespace pkv
