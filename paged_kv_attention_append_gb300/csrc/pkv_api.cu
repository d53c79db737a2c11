// C-ABI entry points (include/pkv.h): argument validation, then kernel
// launches on the caller's stream.  No device allocation happens here.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>

#include "pkv_internal.h"

namespace pkv {

static std::atomic<int64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

constexpr int kMaxDevices = 64;
static std::atomic<int> g_sm_count[kMaxDevices];

int device_sm_count() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices) {
    const int c = g_sm_count[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  if (dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

constexpr int kNumKernelIds = 5;  // PKV_KERNEL_APPEND .. PKV_KERNEL_STATE

struct ProfileEvents {
  void *start[kNumKernelIds] = {};
  void *stop[kNumKernelIds] = {};
};
static thread_local ProfileEvents t_prof;

// While the stream is being captured into a CUDA graph, the record becomes an
// event-record node of the graph (cudaEventRecordExternal), so a replay times
// the kernel with no host launch gap between the event and the kernel.
static void record(void *ev, pkv_stream stream) {
  if (!ev) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(stream, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), stream, cudaEventRecordExternal);
  else
    cudaEventRecord(static_cast<cudaEvent_t>(ev), stream);
}
void profile_begin(int which, pkv_stream stream) { record(t_prof.start[which], stream); }
void profile_end(int which, pkv_stream stream) { record(t_prof.stop[which], stream); }
bool profiling_active() {
  for (int i = 0; i < kNumKernelIds; ++i)
    if (t_prof.start[i] || t_prof.stop[i]) return true;
  return false;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static pkv_status check_pool(const pkv_pool_desc *desc) {
  if (!desc) return PKV_ERR_NULL;
  if (desc->block_size != kBlockSize) return PKV_ERR_UNSUPPORTED;
  if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (desc->num_kv_heads < 1 || desc->num_blocks < 0) return PKV_ERR_SHAPE;
  // TMA row coordinates are int32: rows = num_blocks * 2 * Hkv * 16 must fit.
  if ((int64_t)desc->num_blocks * 2 * desc->num_kv_heads * kBlockSize >= (int64_t)1 << 31)
    return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

extern "C" int32_t pkv_version(void) { return 200; }

extern "C" int64_t pkv_kernel_launch_count(void) { return g_launches.load(); }

extern "C" pkv_status pkv_set_profile_events(int32_t which, void *start_event,
                                             void *stop_event) {
  if (which < 0 || which >= kNumKernelIds) return PKV_ERR_RANGE;
  t_prof.start[which] = start_event;
  t_prof.stop[which] = stop_event;
  return PKV_OK;
}

extern "C" const char *pkv_status_string(int32_t status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: inconsistent sizes";
    case PKV_ERR_RANGE: return "PKV_ERR_RANGE: a length, slot or block id is out of range";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: head_dim/block_size/group not supported";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: plan or workspace buffer too small";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA: a CUDA runtime call failed";
    case PKV_ERR_DEVICE_CHECK: return "PKV_ERR_DEVICE_CHECK: a kernel reported an error";
    case PKV_ERR_ALIGN: return "PKV_ERR_ALIGN: a device pointer is not 16-byte aligned";
    case PKV_ERR_STATE: return "PKV_ERR_STATE: a planner call out of order";
    case PKV_ERR_HOST_MEMORY: return "PKV_ERR_HOST_MEMORY: host memory or a thread for the planner could not be had";
    default: return "unknown pkv status";
  }
}

extern "C" pkv_status pkv_paged_kv_append(const void *k, const void *v,
                                          const int32_t *slot_mapping, int32_t num_tokens,
                                          void *kv_pool, const pkv_pool_desc *desc,
                                          int32_t *dev_status, pkv_stream stream) {
  pkv_status st = check_pool(desc);
  if (st != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !kv_pool) return PKV_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || !aligned16(kv_pool)) return PKV_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(slot_mapping) & 3u) return PKV_ERR_ALIGN;
  int e = launch_append(k, v, slot_mapping, num_tokens, kv_pool, *desc, dev_status, stream);
  return e ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_state_checkpoint(const void *src, const int32_t *dst_slots,
                                           int32_t num_rows, void *pool, int64_t num_slots,
                                           int64_t row_bytes, int32_t *dev_status,
                                           pkv_stream stream) {
  if (num_rows < 0 || num_slots < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return PKV_ERR_SHAPE;
  if (num_rows == 0) return PKV_OK;
  if (!src || !dst_slots || !pool) return PKV_ERR_NULL;
  if (!aligned16(src) || !aligned16(pool) || (reinterpret_cast<uintptr_t>(dst_slots) & 3u))
    return PKV_ERR_ALIGN;
  int e = launch_state_checkpoint(src, dst_slots, num_rows, pool, num_slots, row_bytes,
                                  dev_status, stream);
  return e ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_decode_advance(int32_t *context_lens, int32_t *slot_mapping,
                                         const int32_t *cu_q_lens, const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, int32_t num_seqs,
                                         const pkv_pool_desc *desc, int32_t *dev_status,
                                         pkv_stream stream) {
  pkv_status st = check_pool(desc);
  if (st != PKV_OK) return st;
  if (num_seqs < 0 || max_blocks_per_seq < 0) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!context_lens || !slot_mapping || !cu_q_lens || !block_tables) return PKV_ERR_NULL;
  int e = launch_decode_advance(context_lens, slot_mapping, cu_q_lens, block_tables,
                                max_blocks_per_seq, num_seqs, desc->num_blocks, dev_status, stream);
  return e ? PKV_ERR_CUDA : PKV_OK;
}

extern "C" pkv_status pkv_paged_varlen_attention(
    const void *q, const int32_t *cu_q_lens, const int32_t *context_lens,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const void *kv_pool,
    const pkv_pool_desc *desc, float scale, const pkv_plan_info *info, const void *plan_dev,
    void *out, void *workspace, int64_t workspace_bytes, int32_t *dev_status, pkv_stream stream) {
  pkv_status st = check_pool(desc);
  if (st != PKV_OK) return st;
  if (!info) return PKV_ERR_NULL;
  if (info->num_kv_heads != desc->num_kv_heads || info->head_dim != desc->head_dim ||
      info->num_q_heads < 1 || info->num_q_heads % desc->num_kv_heads != 0)
    return PKV_ERR_SHAPE;
  if (!std::isfinite(scale)) return PKV_ERR_RANGE;
  if (info->num_kernels == 0 || info->total_q == 0) return PKV_OK;
  if (!q || !cu_q_lens || !context_lens || !block_tables || !kv_pool || !plan_dev || !out)
    return PKV_ERR_NULL;
  if (max_blocks_per_seq < info->max_blocks_needed) return PKV_ERR_RANGE;
  if (workspace_bytes < info->workspace_bytes) return PKV_ERR_WORKSPACE;
  if (info->workspace_bytes > 0 && !workspace) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(kv_pool) || !aligned16(plan_dev) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_ALIGN;

  AttnArgs a;
  a.q = q;
  a.out = out;
  a.cu_q_lens = cu_q_lens;
  a.context_lens = context_lens;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.kv_pool = kv_pool;
  a.desc = *desc;
  a.num_q_heads = info->num_q_heads;
  a.num_seqs = info->num_seqs;
  a.total_q = info->total_q;
  a.scale = scale;
  const char *pb = static_cast<const char *>(plan_dev);
  if (info->num_prefill_ctas < 0 || info->num_prefill_ctas > info->num_prefill_tiles ||
      (info->num_prefill_tiles > 0 && info->num_prefill_ctas == 0))
    return PKV_ERR_SHAPE;
  if (info->num_shared_ctas < 0 || info->num_gather_rows < 0 ||
      info->num_shared_items < info->num_shared_ctas * kSharedItemsPerCta)
    return PKV_ERR_SHAPE;
  const PlanOffsets off =
      plan_offsets(info->num_decode_warps, info->num_decode_pieces, info->num_merge_groups,
                   info->num_shared_items, info->num_prefill_tiles, info->num_prefill_ctas,
                   info->num_gather_rows);
  a.warp_begin = reinterpret_cast<const int32_t *>(pb + off.warp_begin);
  a.warp_head = reinterpret_cast<const WarpHead *>(pb + off.warp_head);
  a.num_decode_warps = info->num_decode_warps;
  a.shared_items = reinterpret_cast<const SharedItem *>(pb + off.shared);
  a.num_shared_ctas = info->num_shared_ctas;
  a.num_shared_items = info->num_shared_items;
  a.pieces = reinterpret_cast<const Piece *>(pb + off.pieces);
  a.merge_groups = reinterpret_cast<const MergeGroup *>(pb + off.merges);
  a.num_merge_groups = info->num_merge_groups;
  a.prefill_begin = reinterpret_cast<const int32_t *>(pb + off.prefill_begin);
  a.prefill_tiles = reinterpret_cast<const PrefillTile *>(pb + off.prefill);
  a.gather_rows = reinterpret_cast<const GatherRow *>(pb + off.gather);
  a.num_gather_rows = info->num_gather_rows;
  a.num_partials = info->num_partials;
  a.num_prefill_tiles = info->num_prefill_tiles;
  a.num_prefill_ctas = info->num_prefill_ctas;
  if (info->num_prefill_merges < 0 || info->num_prefill_merges > info->num_merge_groups ||
      info->num_prefill_partials < 0 || info->num_partials < 0)
    return PKV_ERR_SHAPE;
  char *wb = static_cast<char *>(workspace);
  const int d = desc->head_dim;
  const int64_t off_ml = ws_part_o_bytes(info->num_partials, d);
  const int64_t off_po = off_ml + ws_part_ml_bytes(info->num_partials);
  const int64_t off_pml = off_po + ws_ppart_o_bytes(info->num_prefill_partials, d);
  a.part_o = reinterpret_cast<float *>(wb);
  a.part_ml = reinterpret_cast<float *>(wb ? wb + off_ml : nullptr);
  a.ppart_o = reinterpret_cast<float *>(wb ? wb + off_po : nullptr);
  a.ppart_ml = reinterpret_cast<float *>(wb ? wb + off_pml : nullptr);
  a.num_decode_merges = info->num_merge_groups - info->num_prefill_merges;
  a.merge_rows = info->merge_rows;
  if (a.num_decode_merges > 0 && (info->merge_rows < 1 || info->merge_rows > kRowsPerTile))
    return PKV_ERR_SHAPE;
  if (info->lookahead < 0 || (info->lookahead > 0 && info->num_prefill_tiles > 0))
    return PKV_ERR_SHAPE;
  a.lookahead = info->lookahead;
  if (ws_total_bytes(info->num_partials, info->num_prefill_partials, d) > workspace_bytes)
    return PKV_ERR_WORKSPACE;
  a.dev_status = dev_status;
  a.stream = stream;

  if (info->plan_bytes != off.total) return PKV_ERR_SHAPE;
  int launches = 0;
  if (launch_prefill(a, &launches)) return PKV_ERR_CUDA;
  if (launch_decode(a, &launches)) return PKV_ERR_CUDA;
  if (launch_merge(a, &launches)) return PKV_ERR_CUDA;
  return PKV_OK;
}

extern "C" size_t pkv_workspace_size(const pkv_plan_info *info) {
  return info && info->workspace_bytes > 0 ? (size_t)info->workspace_bytes : 0;
}

extern "C" pkv_status pkv_copy_async(void *dst, const void *src, int64_t bytes, pkv_stream stream) {
  if (bytes < 0) return PKV_ERR_RANGE;
  if (bytes == 0) return PKV_OK;
  if (!dst || !src) return PKV_ERR_NULL;
  return cudaMemcpyAsync(dst, src, (size_t)bytes, cudaMemcpyDefault, stream) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_CUDA;
}
