// KV append: scatter this step's K/V rows into their physical pool slots.
//
// The pool is the fixed paged KV store of the vllm-metal page ("Replacing
// attention, reusing the rest"); rows are written in place ("Prefix caching on
// hybrid models": a write touches only the rows it writes, never copies the
// pool).  Pure data movement: each thread moves one 16-byte vector (8 bf16),
// consecutive threads cover consecutive bytes of one (token, K|V, head) row so
// both the loads and the stores are fully coalesced 16-byte accesses.
#include <cuda_runtime.h>

#include "pkv_device.cuh"

namespace pkv {

template <int D>
__global__ void __launch_bounds__(256) append_kernel(const uint4 *__restrict__ k,
                                                     const uint4 *__restrict__ v,
                                                     const int32_t *__restrict__ slot_mapping,
                                                     int32_t num_tokens, uint4 *__restrict__ pool,
                                                     int32_t num_blocks, int32_t hkv,
                                                     int32_t *dev_status) {
  constexpr int kVecPerRow = D / 8;  // 16-byte vectors per head row
  pdl_trigger();  // the attention kernels may launch now; they wait for our writes
  const int64_t per_token = 2ll * hkv * kVecPerRow;
  const int64_t total = per_token * num_tokens;
  const int64_t nslots = (int64_t)num_blocks * kBlockSize;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  // vector idx: its source, and its destination (null: padding token or a bad
  // slot, reported once per token)
  auto locate = [&](int64_t idx, const uint4 *&src, uint4 *&dst) {
    const int32_t t = (int32_t)(idx / per_token);
    int32_t rem = (int32_t)(idx - (int64_t)t * per_token);
    const int32_t kv = rem / (hkv * kVecPerRow);
    rem -= kv * hkv * kVecPerRow;
    const int32_t h = rem / kVecPerRow;
    const int32_t vec = rem - h * kVecPerRow;
    src = (kv == 0 ? k : v) + ((int64_t)t * hkv + h) * kVecPerRow + vec;
    const int64_t slot = __ldg(slot_mapping + t);
    dst = nullptr;
    if (slot >= nslots) {
      if (kv == 0 && h == 0 && vec == 0) report(dev_status, PKV_DEV_BAD_SLOT);
    } else if (slot >= 0) {
      const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
      dst = pool + (((blk * 2 + kv) * hkv + h) * kBlockSize + off) * kVecPerRow + vec;
    }
  };
  // two vectors a thread per round, both loads issued before either store
  for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < total; i0 += 2 * stride) {
    const int64_t i1 = i0 + stride;
    const uint4 *s0, *s1 = nullptr;
    uint4 *d0, *d1 = nullptr;
    locate(i0, s0, d0);
    if (i1 < total) locate(i1, s1, d1);
    const uint4 x0 = d0 ? ldg128_nc(s0) : make_uint4(0, 0, 0, 0);
    const uint4 x1 = d1 ? ldg128_nc(s1) : make_uint4(0, 0, 0, 0);
    if (d0) *d0 = x0;
    if (d1) *d1 = x1;
  }
}

int launch_append(const void *k, const void *v, const int32_t *slot_mapping, int32_t num_tokens,
                  void *kv_pool, const pkv_pool_desc &desc, int32_t *dev_status,
                  pkv_stream stream) {
  const int64_t vecs = 2ll * desc.num_kv_heads * (desc.head_dim / 8) * num_tokens;
  const int threads = 256;
  int64_t blocks = (vecs + threads - 1) / threads;
  // one resident wave at most (8 CTAs of 256 threads per SM), two vectors a
  // thread per round of the grid-stride loop
  const int64_t cap = 8ll * (device_sm_count() > 0 ? device_sm_count() : 1);
  blocks = (blocks + 1) / 2;
  blocks = blocks < 1 ? 1 : (blocks > cap ? cap : blocks);
  const cudaError_t pe = desc.head_dim == 128 ? prepare_kernel<append_kernel<128>>(0)
                                              : prepare_kernel<append_kernel<64>>(0);
  if (pe != cudaSuccess) return (int)pe;
  profile_begin(PKV_KERNEL_APPEND, stream);
  if (desc.head_dim == 128)
    append_kernel<128><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
        static_cast<uint4 *>(kv_pool), desc.num_blocks, desc.num_kv_heads, dev_status);
  else
    append_kernel<64><<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
        static_cast<uint4 *>(kv_pool), desc.num_blocks, desc.num_kv_heads, dev_status);
  profile_end(PKV_KERNEL_APPEND, stream);
  count_launches(1);
  return (int)cudaGetLastError();
}

// Chained decode: moves a decode batch to its next step on the device (the
// vllm-metal page's "Chained greedy decode" keeps the token loop off the CPU).
// One thread per sequence: context += q_len, and the slots of the q_len new
// positions are read from the block table.
__global__ void __launch_bounds__(128) decode_advance_kernel(
    int32_t *__restrict__ context_lens, int32_t *__restrict__ slot_mapping,
    const int32_t *__restrict__ cu_q_lens, const int32_t *__restrict__ block_tables,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t num_blocks, int32_t *dev_status) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= num_seqs) return;
  const int32_t c0 = cu_q_lens[s], q = cu_q_lens[s + 1] - c0;
  if (q <= 0) return;
  const int32_t ctx = context_lens[s] + q;
  context_lens[s] = ctx;
  for (int32_t i = 0; i < q; ++i) {
    const int32_t pos = ctx - q + i, blk = pos / kBlockSize;
    const int32_t phys =
        blk < max_blocks_per_seq ? block_tables[(int64_t)s * max_blocks_per_seq + blk] : -1;
    int32_t slot = -1;
    if (phys >= 0 && phys < num_blocks)
      slot = phys * kBlockSize + pos % kBlockSize;
    else
      report(dev_status, PKV_DEV_BAD_BLOCK);
    slot_mapping[c0 + i] = slot;
  }
}

int launch_decode_advance(int32_t *context_lens, int32_t *slot_mapping, const int32_t *cu_q_lens,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          int32_t num_seqs, int32_t num_blocks, int32_t *dev_status,
                          pkv_stream stream) {
  const cudaError_t pe = prepare_kernel<decode_advance_kernel>(0);
  if (pe != cudaSuccess) return (int)pe;
  decode_advance_kernel<<<(unsigned)((num_seqs + 127) / 128), 128, 0, stream>>>(
      context_lens, slot_mapping, cu_q_lens, block_tables, max_blocks_per_seq, num_seqs,
      num_blocks, dev_status);
  count_launches(1);
  return (int)cudaGetLastError();
}

}  // namespace pkv
