/*
 * Paged KV append + packed varlen attention: CPU reference ("oracle").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes -- the plain definitions, in double precision:
 *
 *  append   (vllm-metal v0.4.0 page, "Replacing attention, reusing the rest":
 *            KV lives in fixed-size pages located by per-request block tables;
 *            "Prefix caching on hybrid models": rows are written in place into
 *            the pool).  For each new token t in order whose slot is >= 0:
 *            block = slot / block_size, offset = slot % block_size, and for every
 *            KV head h the raw 16-bit K row and V row are copied to
 *            pool[block][0][h][offset][:] and pool[block][1][h][offset][:].
 *
 *  attention (same page and section: the step is flattened onto one packed
 *            query axis, cu_seqlens marks request boundaries, one launch covers
 *            prefill chunks, decode tokens and verify windows).  For query row
 *            (token t, query head hq) of sequence s, with i = t - cu[s],
 *            q_s = cu[s+1] - cu[s], ctx = context_lens[s], G = Hq / Hkv and
 *            h = hq / G:
 *              visible keys   p = 0 .. ctx - q_s + i         (causal in chunk)
 *              key p lives at block_tables[s][p / bs], offset p % bs
 *              x_p = scale * sum_d q[t][hq][d] * K[p][h][d]
 *              w_p = exp(x_p - max x) / sum_p' exp(x_p' - max x)
 *              out[t][hq][:] = sum_p w_p * V[p][h][:]
 *
 *  state checkpoint (same page, "Prefix caching on hybrid models": linear-
 *            attention state cannot be addressed by a block table, so reusing a
 *            prefix checkpoints that state at block boundaries, written into the
 *            state pools in place).  For each row i in order whose slot is >= 0,
 *            the row_bytes raw bytes of src row i are copied to pool row slot;
 *            nothing else of the pool changes.
 *
 * Readings where the pages are silent: context_lens includes this step's
 * tokens; the q_s queries are the last q_s positions of the context; KV head of
 * query head hq is hq / G (contiguous groups); a negative slot is padding; a
 * slot or block id outside the pool is an error.
 *
 * bf16 inputs are passed as their raw uint16 bit patterns and widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_ERR_SHAPE = 2, OR_ERR_RANGE = 3 };

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static size_t pool_row(int64_t block, int kv, int h, int off, int hkv, int bs, int d) {
  return ((((size_t)block * 2 + (size_t)kv) * (size_t)hkv + (size_t)h) * (size_t)bs + (size_t)off) *
         (size_t)d;
}

/* Returns the number of tokens skipped because their slot was outside the
 * pool (0 when all slots were valid or padding); those tokens are not written. */
int oracle_paged_kv_append(uint16_t *pool, int num_blocks, int block_size, int num_kv_heads,
                           int head_dim, const uint16_t *k, const uint16_t *v,
                           const int32_t *slot_mapping, int n_tokens) {
  int bad = 0;
  int64_t nslots = (int64_t)num_blocks * block_size;
  for (int t = 0; t < n_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token */
    if (slot >= nslots) { ++bad; continue; }
    int64_t b = slot / block_size;
    int off = (int)(slot % block_size);
    for (int h = 0; h < num_kv_heads; ++h) {
      const uint16_t *ks = k + ((size_t)t * num_kv_heads + h) * head_dim;
      const uint16_t *vs = v + ((size_t)t * num_kv_heads + h) * head_dim;
      memcpy(pool + pool_row(b, 0, h, off, num_kv_heads, block_size, head_dim), ks,
             (size_t)head_dim * sizeof(uint16_t));
      memcpy(pool + pool_row(b, 1, h, off, num_kv_heads, block_size, head_dim), vs,
             (size_t)head_dim * sizeof(uint16_t));
    }
  }
  return bad;
}

/* State-row checkpoint.  Returns the number of rows skipped because their slot
 * was outside the pool (negative slots are skipped silently). */
int64_t oracle_state_checkpoint(uint8_t *pool, int64_t num_slots, int64_t row_bytes,
                                const uint8_t *src, const int32_t *slots, int64_t n_rows) {
  int64_t bad = 0;
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t slot = slots[i];
    if (slot < 0) continue;
    if (slot >= num_slots) { ++bad; continue; }
    memcpy(pool + slot * row_bytes, src + i * row_bytes, (size_t)row_bytes);
  }
  return bad;
}

/* Checks the step metadata; returns OR_OK or an error code. */
int oracle_check_step(int num_seqs, const int32_t *cu_q_lens, const int32_t *context_lens,
                      const int32_t *block_tables, int max_blocks_per_seq, int num_blocks,
                      int block_size) {
  if (num_seqs < 0 || block_size <= 0 || max_blocks_per_seq < 0) return OR_ERR_SHAPE;
  if (num_seqs > 0 && cu_q_lens[0] != 0) return OR_ERR_SHAPE;
  for (int s = 0; s < num_seqs; ++s) {
    int qs = cu_q_lens[s + 1] - cu_q_lens[s];
    int ctx = context_lens[s];
    if (qs < 0) return OR_ERR_SHAPE;
    if (qs > ctx) return OR_ERR_RANGE;
    if (qs == 0) continue;
    int nb = (ctx + block_size - 1) / block_size;
    if (nb > max_blocks_per_seq) return OR_ERR_RANGE;
    for (int j = 0; j < nb; ++j) {
      int32_t b = block_tables[(size_t)s * max_blocks_per_seq + j];
      if (b < 0 || b >= num_blocks) return OR_ERR_RANGE;
    }
  }
  return OR_OK;
}

/* One output row (token t, query head hq) of sequence s; `x` is scratch of at
 * least ctx doubles.  Writes head_dim doubles to `o`. */
static void attend_row(const uint16_t *q, int num_q_heads, const int32_t *cu_q_lens,
                       const int32_t *context_lens, const int32_t *block_tables,
                       int max_blocks_per_seq, const uint16_t *pool, int block_size,
                       int num_kv_heads, int head_dim, double scale, int s, int t, int hq,
                       double *x, double *qd, double *o) {
  int qs = cu_q_lens[s + 1] - cu_q_lens[s];
  int i = t - cu_q_lens[s];
  int ctx = context_lens[s];
  int last = ctx - qs + i; /* last visible key position */
  int group = num_q_heads / num_kv_heads;
  int h = hq / group;
  const int32_t *table = block_tables + (size_t)s * max_blocks_per_seq;
  const uint16_t *qrow = q + ((size_t)t * num_q_heads + hq) * head_dim;
  for (int d = 0; d < head_dim; ++d) qd[d] = widen_bf16(qrow[d]);

  double xmax = -INFINITY;
  for (int p = 0; p <= last; ++p) {
    const uint16_t *kr =
        pool + pool_row(table[p / block_size], 0, h, p % block_size, num_kv_heads, block_size,
                        head_dim);
    double acc = 0.0;
    for (int d = 0; d < head_dim; ++d) acc += qd[d] * widen_bf16(kr[d]);
    x[p] = scale * acc;
    if (x[p] > xmax) xmax = x[p];
  }
  double denom = 0.0;
  for (int p = 0; p <= last; ++p) {
    x[p] = exp(x[p] - xmax);
    denom += x[p];
  }
  for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
  for (int p = 0; p <= last; ++p) {
    const uint16_t *vr =
        pool + pool_row(table[p / block_size], 1, h, p % block_size, num_kv_heads, block_size,
                        head_dim);
    double w = x[p] / denom;
    for (int d = 0; d < head_dim; ++d) o[d] += w * widen_bf16(vr[d]);
  }
}

/*
 * Attention for a list of output rows.  rows[r] = t * num_q_heads + hq; when
 * rows is NULL every row of the step is computed in packed order
 * (n_rows must then equal total_q * num_q_heads).  out: [n_rows][head_dim].
 * num_threads <= 0 uses the OpenMP default.  Returns OR_OK or an error code.
 */
int oracle_paged_varlen_attention(const uint16_t *q, int total_q, int num_q_heads,
                                  const int32_t *cu_q_lens, const int32_t *context_lens,
                                  int num_seqs, const int32_t *block_tables,
                                  int max_blocks_per_seq, const uint16_t *pool, int num_blocks,
                                  int block_size, int num_kv_heads, int head_dim, double scale,
                                  const int64_t *rows, int64_t n_rows, double *out,
                                  int num_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0) return OR_ERR_SHAPE;
  if (num_seqs > 0 && cu_q_lens[num_seqs] != total_q) return OR_ERR_SHAPE;
  int rc = oracle_check_step(num_seqs, cu_q_lens, context_lens, block_tables, max_blocks_per_seq,
                             num_blocks, block_size);
  if (rc != OR_OK) return rc;
  if (rows == NULL && n_rows != (int64_t)total_q * num_q_heads) return OR_ERR_SHAPE;

  /* owner sequence of every packed token */
  int *owner = (int *)malloc(sizeof(int) * (size_t)(total_q > 0 ? total_q : 1));
  int max_ctx = 1;
  for (int s = 0; s < num_seqs; ++s) {
    for (int t = cu_q_lens[s]; t < cu_q_lens[s + 1]; ++t) owner[t] = s;
    if (context_lens[s] > max_ctx) max_ctx = context_lens[s];
  }
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t row = rows ? rows[r] : r;
    if (row < 0 || row >= (int64_t)total_q * num_q_heads) { free(owner); return OR_ERR_RANGE; }
  }

#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
  {
    double *x = (double *)malloc(sizeof(double) * (size_t)max_ctx);
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
    for (int64_t r = 0; r < n_rows; ++r) {
      int64_t row = rows ? rows[r] : r;
      int t = (int)(row / num_q_heads);
      int hq = (int)(row % num_q_heads);
      attend_row(q, num_q_heads, cu_q_lens, context_lens, block_tables, max_blocks_per_seq, pool,
                 block_size, num_kv_heads, head_dim, scale, owner[t], t, hq, x, qd,
                 out + (size_t)r * head_dim);
    }
    free(x);
    free(qd);
  }
  free(owner);
  return OR_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
