// Attention entry point for callers that cannot allocate device memory.
//
// pkv_paged_varlen_attention needs a caller-provided workspace for the fp32
// partial results of row groups whose keys are split over several CTAs.  Some
// callers cannot provide one: code that runs where cudaMalloc is unavailable or
// forbidden (a plugin handed only the step's tensors by a host that owns every
// allocation, a real-time path where an allocation could block or fail, a
// runtime that pre-budgets all device memory).  This entry point gives them the
// same computation with the scratch taken from a fixed array that is part of
// the library's device image instead.
//
// The array is a file-scope static __device__ object: the CUDA driver places it
// in device memory when it loads this library's module on a GPU, and every GPU
// that loads the library keeps those bytes until the process exits.  In host
// code its name is only a host-side stand-in, never a device address, so the
// device address is looked up once per device with cudaGetSymbolAddress.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call made with that device current, then cached).
pkv_status scratch_address(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_paged_varlen_attention_noalloc(
    const void *q, const int32_t *cu_q_lens, const int32_t *context_lens,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const void *kv_pool,
    const pkv_pool_desc *desc, float scale, const pkv_plan_info *info, const void *plan_dev,
    void *out, int32_t *dev_status, pkv_stream stream) {
  if (!info) return PKV_ERR_NULL;
  if (info->workspace_bytes > (int64_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  void *scratch = nullptr;
  pkv_status st = scratch_address(&scratch);
  if (st != PKV_OK) return st;
  return pkv_paged_varlen_attention(q, cu_q_lens, context_lens, block_tables, max_blocks_per_seq,
                                    kv_pool, desc, scale, info, plan_dev, out, scratch,
                                    (int64_t)PKV_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
