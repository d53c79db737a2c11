/*
 * pkv.h -- paged KV cache append and packed varlen attention on one GB300.
 *
 * The problem (vllm-metal v0.4.0 release page, section "Replacing attention,
 * reusing the rest"): a serving step is flattened onto ONE packed query axis,
 * with cu_seqlens marking where each request's query tokens start; KV stays in
 * fixed-size pages located through per-request block tables; one attention
 * launch covers everything the scheduler packed into the step -- chunked
 * prefill chunks, decode tokens and speculative-verify windows.  The same page
 * ("What v0.4.0 adds", batched MTP) has verify windows ride in the packed
 * target batch, and ("Prefix caching on hybrid models") rows are written into
 * pools in place.
 *
 * Conventions shared by every call:
 *  - All tensors are dense and row-major; bf16 is IEEE bfloat16 bit patterns.
 *  - kv_pool:  bf16 [num_blocks][2][num_kv_heads][block_size][head_dim];
 *              index 1 of the second axis selects K (0) or V (1).  Each
 *              (block, K|V, head) slab is one contiguous block_size*head_dim run.
 *  - q, out:   bf16 [total_q][num_q_heads][head_dim], packed in sequence order.
 *  - k, v:     bf16 [num_tokens][num_kv_heads][head_dim] (this step's new tokens).
 *  - cu_q_lens [num_seqs+1] int32, cu_q_lens[0] = 0, non-decreasing;
 *    q_len(s) = cu_q_lens[s+1] - cu_q_lens[s].
 *  - context_lens [num_seqs] int32: keys of sequence s INCLUDING this step's
 *    new tokens (append first, then attend).  q_len(s) <= context_lens[s].
 *  - Causality: query i of sequence s sits at position ctx - q_len + i and sees
 *    keys 0 .. ctx - q_len + i.
 *  - GQA: query head hq reads KV head hq / (num_q_heads / num_kv_heads).
 *  - block_tables [num_seqs][max_blocks_per_seq] int32: logical block j of
 *    sequence s is physical block block_tables[s][j]; entries at or past
 *    ceil(ctx/block_size) are never read.  Several sequences may share blocks.
 *  - Supported: block_size 16, head_dim 64 or 128, num_q_heads a multiple of
 *    num_kv_heads with group size <= 16.  Anything else: PKV_ERR_UNSUPPORTED.
 *
 * Ownership and execution: the caller owns every buffer.  The library never
 * allocates device memory, keeps no per-call state between calls, and enqueues
 * work asynchronously on the caller's stream.  Device pointers must be
 * 16-byte aligned.
 *
 * Errors: host-detectable problems return a non-zero pkv_status before any
 * work is enqueued.  Problems only the device can see (a slot or block id
 * outside the pool, a plan that does not match the device metadata, a pipeline
 * wait that timed out) are written to *dev_status (int32, device memory; first
 * error wins; caller zeroes it and reads it after synchronising); the offending
 * token/block is skipped, nothing is read or written out of bounds, and no
 * kernel traps or asserts.  dev_status may be NULL to ignore them.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *pkv_stream;

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,          /* a required pointer is NULL */
  PKV_ERR_SHAPE = 2,         /* inconsistent sizes (cu_q_lens not monotone, ...) */
  PKV_ERR_RANGE = 3,         /* q_len > context_len, block id / slot out of range, ... */
  PKV_ERR_UNSUPPORTED = 4,   /* head_dim, block_size or group size not supported */
  PKV_ERR_WORKSPACE = 5,     /* plan or workspace buffer too small */
  PKV_ERR_CUDA = 6,          /* a CUDA runtime call failed (launch, attribute, ...) */
  PKV_ERR_DEVICE_CHECK = 7,  /* value written to *dev_status by a kernel */
  PKV_ERR_ALIGN = 8,         /* a device pointer is not 16-byte aligned */
  PKV_ERR_STATE = 9,         /* a call out of order (pkv_planner_post / pkv_planner_wait) */
  PKV_ERR_HOST_MEMORY = 10   /* host memory or a thread for the planner could not be had */
} pkv_status;

/* Device-side error codes written to *dev_status (first one wins). */
#define PKV_DEV_OK 0
#define PKV_DEV_BAD_SLOT 1       /* append: slot >= num_blocks*block_size (token skipped) */
#define PKV_DEV_BAD_BLOCK 2      /* attention: block id outside [0, num_blocks) (block skipped) */
#define PKV_DEV_TIMEOUT 3        /* a pipeline wait exceeded its bound (tile abandoned) */
#define PKV_DEV_PLAN_MISMATCH 4  /* device cu_q_lens/context_lens disagree with the plan */

typedef struct pkv_pool_desc {
  int32_t num_blocks;   /* physical blocks in kv_pool */
  int32_t block_size;   /* tokens per block; must be 16 */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D: 64 or 128 */
} pkv_pool_desc;

/* Summary of a step plan, written by pkv_plan_step. */
typedef struct pkv_plan_info {
  int32_t num_seqs;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t total_q;
  int32_t num_decode_warps;  /* warps of the split-KV kernel; each streams an equal share of keys */
  int32_t num_decode_pieces; /* (row group, KV head, key range) pieces over all decode warps */
  int32_t num_merge_groups;  /* results combined from partials: decode (row group, KV head)
                                pairs whose keys span several pieces, then prefill sub-tiles
                                whose keys span several work items */
  int32_t num_partials;      /* decode partial-result slots (one per piece of a merge group) */
  int32_t num_prefill_tiles; /* tensor-core work items: a key range of two 128-token x 1-head
                                query tiles of one KV head */
  int32_t num_kernels;       /* kernel launches one pkv_paged_varlen_attention call makes */
  int32_t max_blocks_needed; /* max over sequences of ceil(context_len / block_size) */
  int32_t num_prefill_ctas;  /* persistent tensor-core CTAs (one per SM at most); each runs
                                an equal-cost range of the work items' key tiles */
  int32_t num_prefill_partials; /* prefill partial-result slots (128 rows each) */
  int32_t num_prefill_merges;   /* prefill merge groups (the last ones of num_merge_groups) */
  int32_t lookahead;            /* further decode steps the plan stays valid for (chained
                                   decode, pkv_plan_decode_chain); 0 for a single step */
  int32_t num_shared_ctas;      /* split-KV CTAs whose warp pairs each read blocks several row
                                   groups share once for two of them: a prefix several
                                   sequences share (needs host block tables), or a verify
                                   window wider than one row group */
  int32_t num_gather_rows;      /* query tokens listed by the tensor-core shared-prefix
                                   items (a prefix many query rows share is read once per
                                   128 rows on the tensor cores; needs host block tables) */
  int32_t merge_rows;           /* query rows of the largest decode merge group (its row
                                   group's tokens x the G heads of a KV head, <= 16; 0 when
                                   there is none): the merge launch covers that many rows
                                   of every decode group */
  int32_t num_shared_items;     /* shared-block items of those CTAs' warp pairs (each pair
                                   runs a chain of them, one after another) */
  int64_t kv_tokens;         /* sum of context_lens over sequences with q_len > 0 */
  int64_t decode_blocks;     /* (KV block, KV head) pairs the split-KV kernel attends, each
                                counted once: per sequence (however many row groups read
                                it), a prefix its shared-prefix CTAs read once per group,
                                a prefix gathered onto the tensor cores not at all */
  int64_t plan_bytes;        /* bytes of the plan buffer (host, then device copy) */
  int64_t workspace_bytes;   /* device workspace the attention call needs */
  int64_t gather_pairs;      /* (query row, key) pairs the tensor-core kernel computes for
                                gathered shared-prefix rows (row = token x query head) */
} pkv_plan_info;

/* Library version (major*10000 + minor*100 + patch). */
PKV_API int32_t pkv_version(void);

/* Human-readable name of a pkv_status or a PKV_DEV_* code. */
PKV_API const char *pkv_status_string(int32_t status);

/* Total kernel launches enqueued by this library since it was loaded. */
PKV_API int64_t pkv_kernel_launch_count(void);

/* Kernel ids for pkv_set_profile_events. */
#define PKV_KERNEL_APPEND 0
#define PKV_KERNEL_DECODE 1
#define PKV_KERNEL_MERGE 2
#define PKV_KERNEL_PREFILL 3
#define PKV_KERNEL_STATE 4

/*
 * Profiling hook (off by default).  After this call, every launch of kernel
 * `which` made FROM THE CALLING HOST THREAD is bracketed by
 * cudaEventRecord(start_event) / cudaEventRecord(stop_event) on the launch
 * stream, so the caller can time that kernel alone with its own events
 * (cudaEvent_t handles, created and owned by the caller).  When the launch
 * stream is being captured into a CUDA graph the records are made with
 * cudaEventRecordExternal, i.e. they become event-record nodes that fire on
 * every replay.  While any event is set, kernels launch without programmatic
 * dependent launch, so each one's interval holds that kernel alone.  Passing
 * NULL for both turns it off again.  Returns PKV_ERR_RANGE for an unknown
 * kernel id.
 */
PKV_API pkv_status pkv_set_profile_events(int32_t which, void *start_event, void *stop_event);

/*
 * KV append (the in-place row scatter of the "Prefix caching on hybrid
 * models" section, applied to the paged KV pool of "Replacing attention,
 * reusing the rest").
 *   For each token t < num_tokens with slot = slot_mapping[t]:
 *     slot < 0                        : padding, nothing written;
 *     0 <= slot < num_blocks*bs       : kv_pool[slot/bs][0][h][slot%bs][:] = k[t][h][:],
 *                                       kv_pool[slot/bs][1][h][slot%bs][:] = v[t][h][:]
 *                                       for every KV head h (raw 16-bit copies);
 *     slot >= num_blocks*bs           : token skipped, PKV_DEV_BAD_SLOT to *dev_status.
 *   k, v: device bf16 [num_tokens][Hkv][D]; slot_mapping: device int32 [num_tokens];
 *   kv_pool: device, layout above.  Two tokens with the same slot: unspecified
 *   which one lands.  num_tokens == 0 enqueues nothing and returns PKV_OK.
 */
PKV_API pkv_status pkv_paged_kv_append(const void *k, const void *v, const int32_t *slot_mapping,
                               int32_t num_tokens, void *kv_pool, const pkv_pool_desc *desc,
                               int32_t *dev_status, pkv_stream stream);

/*
 * Host step metadata (the per-threadgroup search over cu_seqlens that the
 * vllm-metal kernel performs, moved to the host where the scheduler already
 * holds the lengths).  Validates the lengths, splits each sequence's keys into
 * work tiles sized for num_sms SMs, assigns partial-result slots and sizes the
 * workspace.
 *   cu_q_lens, context_lens: HOST arrays (num_seqs+1 and num_seqs int32).
 *   num_sms: SMs of the target GPU; <= 0 asks the CUDA runtime for the SM count
 *   of the calling thread's current device (PKV_ERR_CUDA if there is none).
 *   plan: host buffer receiving plan_capacity bytes at most; may be NULL to
 *   query sizes only (info is always filled on success).
 * Returns PKV_ERR_WORKSPACE if plan is non-NULL and plan_capacity < info->plan_bytes,
 * PKV_ERR_HOST_MEMORY if the planner's own host scratch (reused per calling
 * thread, grown with the step) could not be allocated.
 * The plan buffer is opaque; upload it unchanged (e.g. cudaMemcpyAsync) before
 * the attention call that uses it.
 *
 * Compared with the plainest form of this call -- (cu_q_lens, context_lens,
 * num_seqs, num_q_heads, pool) -> plan -- three things are added, each because
 * the plan depends on it or the caller should own it: num_sms (the work is cut
 * into equal shares for that many SMs, so a plan is tied to a GPU size); a
 * caller-owned plan buffer with its capacity (the library allocates nothing,
 * host or device, and the caller picks pinned memory for an asynchronous
 * upload); and the pkv_plan_info summary, which the attention call takes in
 * place of parsing the device copy of the plan on the host.
 */
PKV_API pkv_status pkv_plan_step(const int32_t *cu_q_lens, const int32_t *context_lens, int32_t num_seqs,
                         int32_t num_q_heads, const pkv_pool_desc *desc, int32_t num_sms,
                         void *plan, int64_t plan_capacity, pkv_plan_info *info);

/*
 * Host planning on a worker thread.  A serving loop plans each step on the host
 * while it also queues that step's input copy and KV append (the append needs
 * no plan); with the planner on a thread of its own, the plan is computed while
 * the calling thread issues those calls instead of after them.  A pkv_planner
 * owns one thread and runs one pkv_plan_step_ex call at a time.
 *
 * pkv_planner_create: starts the thread.  After finishing a job the thread
 * polls for the next one for spin_us microseconds (so a loop whose steps follow
 * each other within that time hands a job over without a thread wake-up), then
 * sleeps until one is posted; spin_us <= 0 sleeps at once.  *out receives the
 * planner.  Errors: PKV_ERR_NULL (out NULL), PKV_ERR_RANGE (spin_us above
 * 1,000,000), PKV_ERR_HOST_MEMORY (the planner or its thread could not be
 * created).
 *
 * pkv_planner_destroy: finishes a posted job, stops and joins the thread and
 * frees the planner.  NULL is a no-op.  Not to be called concurrently with
 * another call on the same planner.
 *
 * pkv_planner_post: hands the thread one pkv_plan_step_ex call with these
 * arguments and returns at once.  Every pointer must stay valid, and the arrays
 * and *desc unchanged, until pkv_planner_wait has returned; the thread writes
 * plan and *info.  num_sms <= 0 is resolved here, on the calling thread's
 * current device (PKV_ERR_CUDA if there is none), not on the worker.
 * PKV_ERR_STATE if a job is already posted and not yet waited for; PKV_ERR_NULL
 * if planner is NULL.  The job's own errors come from pkv_planner_wait.  The
 * thread keeps its own planner scratch, as any calling thread does.
 *
 * pkv_planner_wait: waits (polling) until the posted job has finished and
 * returns its status, the value pkv_plan_step_ex would have returned; *info
 * and the plan buffer then hold its results.  PKV_ERR_STATE if no job is
 * posted; PKV_ERR_NULL if planner is NULL.
 *
 * post and wait on one planner are meant for one calling thread at a time.
 */
typedef struct pkv_planner pkv_planner;
PKV_API pkv_status pkv_planner_create(int32_t spin_us, pkv_planner **out);
PKV_API void pkv_planner_destroy(pkv_planner *planner);
PKV_API pkv_status pkv_planner_post(pkv_planner *planner, const int32_t *cu_q_lens,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, const pkv_pool_desc *desc,
                                    int32_t num_sms, int32_t steps, const int32_t *block_tables,
                                    int32_t max_blocks_per_seq, int32_t prefill_min_q, void *plan,
                                    int64_t plan_capacity, pkv_plan_info *info);
PKV_API pkv_status pkv_planner_wait(pkv_planner *planner);

/*
 * Bytes of device workspace the attention call needs for a plan (the same
 * value as info->workspace_bytes; 0 when the step needs none).  info NULL: 0.
 */
PKV_API size_t pkv_workspace_size(const pkv_plan_info *info);

/*
 * Stream-ordered copy of `bytes` bytes from src to dst on `stream`, for moving
 * a step's inputs and plan up and its output back without leaving this API:
 * host to device, device to host or device to device, the direction taken from
 * the pointers (unified addressing).  The call returns once the copy is queued;
 * it is asynchronous with respect to the host only when the host side is pinned
 * (page-locked) memory, and the caller keeps both buffers alive and unchanged
 * until the stream has passed the copy.  bytes == 0: nothing is queued.
 * Errors: PKV_ERR_RANGE (bytes < 0), PKV_ERR_NULL (a NULL pointer with
 * bytes > 0), PKV_ERR_CUDA (the runtime refused the copy).
 */
PKV_API pkv_status pkv_copy_async(void *dst, const void *src, int64_t bytes, pkv_stream stream);

/*
 * Plan for a chain of `steps` decode steps of the same batch (the vllm-metal
 * page's MLX engine, "Chained greedy decode": several decode steps built into
 * one graph and run with a single sync per chunk).  context_lens are those of
 * the first step; every later step adds each sequence's q_len tokens.  The one
 * plan serves all steps: it is sized for the last step's contexts, and each
 * step reads the current contexts from the device copy of context_lens, which
 * pkv_decode_advance moves on between steps.  Block tables must already hold
 * the blocks of the last step's contexts (info->max_blocks_needed counts them).
 * Sequences with q_len >= 64 (tensor-core prefill rows) are not supported here:
 * PKV_ERR_UNSUPPORTED.  steps < 1: PKV_ERR_RANGE.  Otherwise as pkv_plan_step;
 * info->lookahead = steps - 1.
 */
PKV_API pkv_status pkv_plan_decode_chain(const int32_t *cu_q_lens, const int32_t *context_lens,
                                         int32_t num_seqs, int32_t num_q_heads,
                                         const pkv_pool_desc *desc, int32_t num_sms, int32_t steps,
                                         void *plan, int64_t plan_capacity, pkv_plan_info *info);

/*
 * The general form of pkv_plan_step / pkv_plan_decode_chain: steps = 1 is a
 * single step, steps > 1 a decode chain.  block_tables, when not NULL, is a
 * HOST copy of the step's block tables ([num_seqs][max_blocks_per_seq] int32,
 * the same entries the device copy holds): the plan then also carries the
 * physical ids of the first blocks each split-KV warp reads, so its first copies
 * start without waiting for a block-table read, and sequences whose tables
 * start with the same physical blocks read those blocks once per work unit.
 * The attention kernel checks the carried ids against the device block tables;
 * on a disagreement it reports PKV_DEV_PLAN_MISMATCH and writes no result built
 * from the disagreeing blocks (those rows of out are left as they were).
 * prefill_min_q: sequences with at least this many query tokens run on the
 * tensor-core prefill kernel; 0 picks the default (64); a negative value keeps
 * every sequence on the split-KV kernel (both compute the same function).
 */
PKV_API pkv_status pkv_plan_step_ex(const int32_t *cu_q_lens, const int32_t *context_lens,
                                    int32_t num_seqs, int32_t num_q_heads,
                                    const pkv_pool_desc *desc, int32_t num_sms, int32_t steps,
                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                    int32_t prefill_min_q, void *plan, int64_t plan_capacity,
                                    pkv_plan_info *info);

/*
 * Device-side move to the next step of a decode chain: for every sequence s
 * with q = cu_q_lens[s+1] - cu_q_lens[s] > 0, context_lens[s] += q and
 * slot_mapping[cu_q_lens[s] + i] = the pool slot of position
 * context_lens[s] - q + i (new value), i.e. block_tables[s][pos / block_size] *
 * block_size + pos % block_size, for i < q.  A position whose block lies
 * outside the table or the pool gets slot -1 (not written by the next append)
 * and PKV_DEV_BAD_BLOCK goes to *dev_status.  All arrays are device int32;
 * the kernel runs after the preceding attention call in stream order, so that
 * call read the old contexts.
 */
PKV_API pkv_status pkv_decode_advance(int32_t *context_lens, int32_t *slot_mapping,
                                      const int32_t *cu_q_lens, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, int32_t num_seqs,
                                      const pkv_pool_desc *desc, int32_t *dev_status,
                                      pkv_stream stream);

/*
 * Packed varlen attention over the paged KV pool ("Replacing attention,
 * reusing the rest": one launch sequence for prefill chunks, decode tokens and
 * verify windows):
 *   out[t][hq][:] = sum_p softmax_p(scale * q[t][hq] . K[p][hq/G]) V[p][hq/G]
 *   over the keys p visible to token t (causal rule above), K/V of position p
 *   read from kv_pool block block_tables[s][p/bs], offset p%bs.
 *   q, out: device bf16 (layout above).  cu_q_lens, context_lens, block_tables:
 *   DEVICE copies of the arrays the plan was built from.  plan_dev: device copy
 *   of the plan buffer; info: the host summary pkv_plan_step returned.
 *   workspace: device scratch of at least info->workspace_bytes (256-byte
 *   aligned; contents on entry do not matter).  Rows of sequences with
 *   q_len == 0 do not exist.  Accumulation is fp32; out is rounded once to bf16.
 *   Kernels are launched with programmatic stream serialisation: their launch
 *   overlaps the tail of the preceding kernel on the stream.  The first kernel
 *   of the call waits for that preceding kernel to complete
 *   (griddepcontrol.wait) before it reads kv_pool or the workspace; the plan,
 *   q, cu_q_lens, context_lens and block_tables are read before that wait.  A
 *   kernel that lets its dependents launch early
 *   (griddepcontrol.launch_dependents) and runs right before this call must
 *   therefore not write those five: this library's KV append writes only
 *   kv_pool; kernels that do not signal early are simply waited for.  Inside
 *   the call, when a step has both tensor-core and split-KV work, the
 *   tensor-core kernel lets the split-KV kernel launch only once its own wait
 *   has returned, so the split-KV kernel reads the pool without a further wait
 *   and starts on each SM the tensor-core kernel's persistent CTAs leave; it
 *   waits at its end instead, so every kernel of the call completes after the
 *   ones before it (the call as a whole is stream-ordered).
 */
PKV_API pkv_status pkv_paged_varlen_attention(const void *q, const int32_t *cu_q_lens,
                                      const int32_t *context_lens, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const void *kv_pool,
                                      const pkv_pool_desc *desc, float scale,
                                      const pkv_plan_info *info, const void *plan_dev, void *out,
                                      void *workspace, int64_t workspace_bytes,
                                      int32_t *dev_status, pkv_stream stream);

/*
 * State-row checkpoint (the vllm-metal v0.4.0 page, "Prefix caching on hybrid
 * models"): linear-attention layers keep a recurrent state per sequence that a
 * block table cannot address, so reusing a prefix means checkpointing that
 * state at block boundaries into state pools, and the rows are written in place
 * rather than by copying the pool.
 *   For each row i < num_rows with slot = dst_slots[i]:
 *     slot < 0               : nothing written;
 *     0 <= slot < num_slots  : pool[slot][0 .. row_bytes) = src[i][0 .. row_bytes)
 *                              (raw bytes);
 *     slot >= num_slots      : row skipped, PKV_DEV_BAD_SLOT to *dev_status.
 *   src: device [num_rows][row_bytes]; dst_slots: device int32 [num_rows];
 *   pool: device [num_slots][row_bytes].  row_bytes must be a positive multiple
 *   of 16 (else PKV_ERR_SHAPE) and src, pool 16-byte aligned (else
 *   PKV_ERR_ALIGN).  Bytes outside the written rows are untouched.  Two rows
 *   with the same slot: unspecified which one lands.  num_rows == 0 enqueues
 *   nothing and returns PKV_OK.
 */
PKV_API pkv_status pkv_state_checkpoint(const void *src, const int32_t *dst_slots,
                                        int32_t num_rows, void *pool, int64_t num_slots,
                                        int64_t row_bytes, int32_t *dev_status,
                                        pkv_stream stream);

/*
 * Size of the fixed scratch array used by pkv_paged_varlen_attention_noalloc
 * (16 MiB).  Every GPU that loads this library holds these bytes until the
 * process exits.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16 * 1024 * 1024)

/*
 * pkv_paged_varlen_attention without a workspace argument, for callers that
 * cannot allocate device memory (no cudaMalloc available or allowed: a plugin
 * that is handed only the step's tensors, a path where an allocation could
 * block or fail, a runtime that pre-budgets all device memory).  The pages have
 * no counterpart to this call; it exists only for such callers.
 *
 * Same arguments, computation and results as pkv_paged_varlen_attention; the
 * caller still passes every input and the output.  The split-KV partial
 * results go to a fixed array in the library's device image
 * (PKV_NOALLOC_SCRATCH_BYTES), so this call allocates nothing: no cudaMalloc,
 * no cudaFree, no allocating library routine.
 *  - Returns PKV_ERR_WORKSPACE, before anything is enqueued, when the step
 *    needs more scratch than that (info->workspace_bytes >
 *    PKV_NOALLOC_SCRATCH_BYTES); plan such steps with more SMs' worth of
 *    smaller splits or use pkv_paged_varlen_attention.
 *  - The calling thread's current device must be the device of the buffers and
 *    the stream.  The first call made with a given device current looks up the
 *    array's device address on that device (cudaGetSymbolAddress, which may
 *    load the library's module there); make that first call before any stream
 *    capture.  The address is kept for the life of the loaded library: after
 *    cudaDeviceReset on a device, do not call this entry point on that device
 *    again in the same process (the kept address would be stale).
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents.  Nothing in it needs to start at zero (every partial is written
 *    before it is read).  Calls whose work overlaps on the GPU (different
 *    streams, or different host threads, without ordering between them) race
 *    on the array and give wrong results: order them on one stream.
 */
PKV_API pkv_status pkv_paged_varlen_attention_noalloc(
    const void *q, const int32_t *cu_q_lens, const int32_t *context_lens,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const void *kv_pool,
    const pkv_pool_desc *desc, float scale, const pkv_plan_info *info, const void *plan_dev,
    void *out, int32_t *dev_status, pkv_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
