// State-row checkpoint: in-place row writes into a state pool.
//
// The vllm-metal page ("Prefix caching on hybrid models") explains why this
// exists: gated-delta-net linear-attention layers carry a recurrent state that
// a block table cannot address, so reusing a prefix means checkpointing that
// state at block boundaries into state pools (about 1.6 GiB each once ~1,650
// blocks are cached), and the page's fix writes those rows in place instead of
// copying the whole pool first.  Here that is a scatter of whole rows: row i of
// src goes to pool row dst_slots[i]; nothing else of the pool is touched.
//
// Pure data movement, HBM-bound: every thread moves 16-byte vectors, consecutive
// threads cover consecutive bytes of a row (coalesced loads and stores), several
// vectors per thread are in flight before any is stored, and the stores are
// streaming (a checkpoint is not read back soon).
#include <cuda_runtime.h>

#include "pkv_device.cuh"

namespace pkv {

namespace {

constexpr int kStateThreads = 256;
constexpr int kStateUnroll = 4;

__global__ void __launch_bounds__(kStateThreads)
    state_checkpoint_kernel(const uint4 *__restrict__ src, const int32_t *__restrict__ slots,
                            int64_t total_vecs, int64_t vecs_per_row, uint4 *__restrict__ pool,
                            int64_t num_slots, int32_t *dev_status) {
  const int64_t stride = (int64_t)gridDim.x * kStateThreads;
  for (int64_t base = (int64_t)blockIdx.x * kStateThreads + threadIdx.x; base < total_vecs;
       base += stride * kStateUnroll) {
    uint4 v[kStateUnroll];
    int64_t dst[kStateUnroll];
#pragma unroll
    for (int u = 0; u < kStateUnroll; ++u) {
      const int64_t idx = base + u * stride;
      dst[u] = -1;
      if (idx < total_vecs) {
        const int64_t row = idx / vecs_per_row, col = idx - row * vecs_per_row;
        const int64_t slot = __ldg(slots + row);
        if (slot >= 0 && slot < num_slots) {
          dst[u] = slot * vecs_per_row + col;
          v[u] = ldg128_nc(src + idx);
        } else if (slot >= num_slots && col == 0) {
          report(dev_status, PKV_DEV_BAD_SLOT);  // row skipped
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kStateUnroll; ++u)
      if (dst[u] >= 0) __stcs(pool + dst[u], v[u]);
  }
}

}  // namespace

int launch_state_checkpoint(const void *src, const int32_t *dst_slots, int32_t num_rows,
                            void *pool, int64_t num_slots, int64_t row_bytes, int32_t *dev_status,
                            pkv_stream stream) {
  const int64_t vecs_per_row = row_bytes / 16;
  const int64_t total = vecs_per_row * num_rows;
  int64_t blocks = (total + (int64_t)kStateThreads * kStateUnroll - 1) /
                   ((int64_t)kStateThreads * kStateUnroll);
  // a grid-stride loop: at most 8 CTAs per SM
  const int64_t cap = 8ll * (device_sm_count() > 0 ? device_sm_count() : 1);
  blocks = blocks < 1 ? 1 : (blocks > cap ? cap : blocks);
  const cudaError_t pe = prepare_kernel<state_checkpoint_kernel>(0);
  if (pe != cudaSuccess) return (int)pe;
  profile_begin(PKV_KERNEL_STATE, stream);
  state_checkpoint_kernel<<<(unsigned)blocks, kStateThreads, 0, stream>>>(
      static_cast<const uint4 *>(src), dst_slots, total, vecs_per_row, static_cast<uint4 *>(pool),
      num_slots, dev_status);
  profile_end(PKV_KERNEL_STATE, stream);
  count_launches(1);
  return (int)cudaGetLastError();
}

}  // namespace pkv
