/*
 * Plain fp64 CPU oracle for MLA decode attention over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link,
 * load or call this file.  It exists so that the tests, the smoke check and
 * the CPU baseline leg of the benchmark can compare the CUDA kernels against
 * an obviously correct statement of what they compute.  It shares no code,
 * header, table or helper with the CUDA library.
 *
 * What it computes (the definition, written out):
 *   FlashMLA "flash_mla_with_kvcache" as benchmarked in the PAI tutorial
 *   ("云上玩转DeepSeek系列之五", section 4 "不同 MLA 实现的简易性能比较",
 *   the compare_a benchmark): q[b, s_q, h_q, d], a paged cache
 *   blocked_k[num_blocks, block_size, h_kv, d] addressed through
 *   block_table[b, max_blocks], per-sequence cache_seqlens[b], value width dv,
 *   an optional causal mask, outputs out[b, s_q, h_q, dv] and lse[b, h_q, s_q].
 *
 *   For a sequence i, query position j and query head h, with
 *   g = h / (h_q / h_kv) the latent KV head it reads:
 *     visible tokens t:  0 <= t < L_i                     (non-causal)
 *                        0 <= t <= L_i - s_q + j          (causal, the query
 *                        block sits at the end of the sequence)
 *     K_t   = blocked_k[block_table[i][t / block_size]][t % block_size][g][0:d]
 *     V_t   = K_t[0:dv]             (the value is the leading dv latent dims)
 *     s_t   = scale * <q[i,j,h,:], K_t>
 *     lse   = ln sum_t exp(s_t)     (natural log; evaluated as max + log of
 *                                    the shifted sum so that it cannot overflow)
 *     out   = sum_t exp(s_t - lse) * V_t
 *   A row with no visible token gets out = 0 and lse = -inf.
 *
 * The entry stride (elements between consecutive cache entries) is an
 * argument, so the 576-element layout and the 256-byte aligned 640-element
 * layout of vLLM PR #12676 ("Mem align KV caches for CUDA devices") are read
 * through the same code; only the first d elements of an entry are used.
 *
 * Every floating-point step is fp64 from exactly converted bf16 inputs.
 * Work is spread over POSIX threads by output row; each row is computed by
 * one thread with a fixed summation order, so results do not depend on the
 * thread count.
 *
 * Parity status: pinned.  The tests check this file against a dense NumPy
 * brute force on tiny inputs, hand-derived closed forms (single token,
 * all-equal scores, one dominant key, a two-token case) and the invariants of
 * the definition (page permutation, split-and-merge by LSE, entry stride,
 * causal equivalences, head equivariance).  Deliberately broken variants
 * (the `mutation` argument below, used only by those tests) must fail them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Mutations: planted mistakes for the tests that prove the pins can fail.
 * 0 is the oracle itself. */
enum {
  MUT_NONE = 0,
  MUT_DROP_LAST_TOKEN = 1,   /* forgets the last visible token            */
  MUT_CAUSAL_OFF_BY_ONE = 2, /* lets each causal query see one more key   */
  MUT_V_OFFSET = 3,          /* takes V from dims [d - dv, d)             */
  MUT_NO_SCALE = 4,          /* ignores softmax_scale                     */
  MUT_IGNORE_BLOCK_TABLE = 5,/* reads pages linearly, not via block_table */
  MUT_LSE_BASE2 = 6,         /* reports lse in base 2                     */
  MUT_HEAD_GROUP = 7,        /* maps head h to KV head h % h_kv           */
  MUT_ROPE_DROPPED = 8,      /* scores use only the first dv dims         */
  MUT_COUNT = 9
};

static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

typedef struct {
  const uint16_t *q;
  int b, s_q, h_q, d;
  const uint16_t *kcache;
  int64_t num_blocks;
  int block_size, h_kv, stride;
  const int32_t *block_table;
  int max_blocks_per_seq;
  const int32_t *cache_seqlens;
  int dv;
  double scale;
  int causal;
  const int32_t *rows; /* n_rows x 3 (i, j, h) */
  int64_t n_rows;
  double *out; /* n_rows x dv */
  double *lse; /* n_rows      */
  int mutation;
  int64_t next_row; /* shared work counter, taken with an atomic add */
  int error;        /* set by a worker on an invalid page id */
} oracle_job;

/* Address of entry (token t of sequence i, KV head g), or NULL if the page id
 * is outside the cache. */
static const uint16_t *entry_of(const oracle_job *J, int i, int t, int g) {
  int page_slot = t / J->block_size;
  int64_t page = J->mutation == MUT_IGNORE_BLOCK_TABLE
                     ? (int64_t)i * J->max_blocks_per_seq + page_slot
                     : (int64_t)J->block_table[(int64_t)i * J->max_blocks_per_seq + page_slot];
  if (page < 0 || page >= J->num_blocks) return NULL;
  int64_t entry = (page * J->block_size + (t % J->block_size)) * J->h_kv + g;
  return J->kcache + entry * J->stride;
}

static void one_row(oracle_job *J, int64_t r, double *scores) {
  int i = J->rows[3 * r + 0], j = J->rows[3 * r + 1], h = J->rows[3 * r + 2];
  double *out = J->out + r * J->dv;
  int heads_per_kv = J->h_q / J->h_kv;
  int g = J->mutation == MUT_HEAD_GROUP ? h % J->h_kv : h / heads_per_kv;
  int L = J->cache_seqlens[i];

  int visible = L;
  if (J->causal) {
    visible = L - J->s_q + j + 1;
    if (J->mutation == MUT_CAUSAL_OFF_BY_ONE) visible += 1;
  }
  if (visible > L) visible = L;
  if (J->mutation == MUT_DROP_LAST_TOKEN && visible > 0) visible -= 1;

  for (int c = 0; c < J->dv; ++c) out[c] = 0.0;
  if (visible <= 0) {
    J->lse[r] = -INFINITY;
    return;
  }

  const uint16_t *qrow =
      J->q + (((int64_t)i * J->s_q + j) * J->h_q + h) * (int64_t)J->d;
  double scale = J->mutation == MUT_NO_SCALE ? 1.0 : J->scale;
  int score_dims = J->mutation == MUT_ROPE_DROPPED ? J->dv : J->d;

  /* s_t = scale * <q, K_t> */
  double mx = -INFINITY;
  for (int t = 0; t < visible; ++t) {
    const uint16_t *k = entry_of(J, i, t, g);
    if (!k) {
      J->error = 1;
      J->lse[r] = NAN;
      return;
    }
    double dot = 0.0;
    for (int c = 0; c < score_dims; ++c)
      dot += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(k[c]);
    scores[t] = scale * dot;
    if (scores[t] > mx) mx = scores[t];
  }

  /* lse = ln sum_t exp(s_t), as max + ln sum exp(s_t - max) */
  double sum = 0.0;
  for (int t = 0; t < visible; ++t) sum += exp(scores[t] - mx);
  double lse = mx + log(sum);

  /* out = sum_t exp(s_t - lse) V_t,  V_t = K_t[0:dv] */
  int v_off = J->mutation == MUT_V_OFFSET ? J->d - J->dv : 0;
  for (int t = 0; t < visible; ++t) {
    const uint16_t *k = entry_of(J, i, t, g);
    double w = exp(scores[t] - lse);
    for (int c = 0; c < J->dv; ++c) out[c] += w * bf16_bits_to_double(k[v_off + c]);
  }
  J->lse[r] = J->mutation == MUT_LSE_BASE2 ? lse / log(2.0) : lse;
}

static void *worker_main(void *arg) {
  oracle_job *J = (oracle_job *)arg;
  int max_L = 0;
  for (int i = 0; i < J->b; ++i)
    if (J->cache_seqlens[i] > max_L) max_L = J->cache_seqlens[i];
  double *scores = (double *)malloc(sizeof(double) * (size_t)(max_L > 0 ? max_L : 1));
  if (!scores) {
    J->error = 2;
    return NULL;
  }
  for (;;) {
    int64_t r = __atomic_fetch_add(&J->next_row, 1, __ATOMIC_RELAXED);
    if (r >= J->n_rows) break;
    one_row(J, r, scores);
  }
  free(scores);
  return NULL;
}

/*
 * Computes the rows listed in `rows` (n_rows triples i, j, h).
 * q, kcache: bf16 bit patterns.  kcache holds num_blocks * block_size * h_kv
 * entries of `stride` elements each.  out: n_rows x dv doubles, lse: n_rows.
 * Returns 0 on success, 1 if a visible token's page id is outside
 * [0, num_blocks), 2 on allocation failure, -1 on bad arguments.
 */
int mla_oracle_rows_mutant(const uint16_t *q, int b, int s_q, int h_q, int d,
                           const uint16_t *kcache, int64_t num_blocks, int block_size,
                           int h_kv, int stride, const int32_t *block_table,
                           int max_blocks_per_seq, const int32_t *cache_seqlens, int dv,
                           double softmax_scale, int causal, const int32_t *rows,
                           int64_t n_rows, double *out, double *lse, int n_threads,
                           int mutation) {
  if (b <= 0 || s_q <= 0 || h_q <= 0 || h_kv <= 0 || h_q % h_kv != 0 || d <= 0 ||
      dv <= 0 || dv > d || stride < d || block_size <= 0 || n_rows < 0 ||
      mutation < 0 || mutation >= MUT_COUNT)
    return -1;
  for (int64_t r = 0; r < n_rows; ++r) {
    int i = rows[3 * r], j = rows[3 * r + 1], h = rows[3 * r + 2];
    if (i < 0 || i >= b || j < 0 || j >= s_q || h < 0 || h >= h_q) return -1;
  }
  for (int i = 0; i < b; ++i) {
    if (cache_seqlens[i] < 0 ||
        (int64_t)cache_seqlens[i] > (int64_t)max_blocks_per_seq * block_size)
      return -1;
  }
  if (n_threads < 1) n_threads = 1;
  if (n_threads > 512) n_threads = 512;

  oracle_job J = {q,     b,          s_q,           h_q,
                  d,     kcache,     num_blocks,    block_size,
                  h_kv,  stride,     block_table,   max_blocks_per_seq,
                  cache_seqlens, dv, softmax_scale, causal,
                  rows,  n_rows,     out,           lse,
                  mutation, 0, 0};
  /* Rows are handed out through a shared counter; a thread that fails to
   * start simply leaves its share to the others. */
  pthread_t th[512];
  int started[512];
  for (int t = 1; t < n_threads; ++t)
    started[t] = pthread_create(&th[t], NULL, worker_main, &J) == 0;
  worker_main(&J);
  for (int t = 1; t < n_threads; ++t)
    if (started[t]) pthread_join(th[t], NULL);
  return J.error;
}

int mla_oracle_rows(const uint16_t *q, int b, int s_q, int h_q, int d,
                    const uint16_t *kcache, int64_t num_blocks, int block_size, int h_kv,
                    int stride, const int32_t *block_table, int max_blocks_per_seq,
                    const int32_t *cache_seqlens, int dv, double softmax_scale, int causal,
                    const int32_t *rows, int64_t n_rows, double *out, double *lse,
                    int n_threads) {
  return mla_oracle_rows_mutant(q, b, s_q, h_q, d, kcache, num_blocks, block_size, h_kv,
                                stride, block_table, max_blocks_per_seq, cache_seqlens, dv,
                                softmax_scale, causal, rows, n_rows, out, lse, n_threads,
                                MUT_NONE);
}

int mla_oracle_mutation_count(void) { return MUT_COUNT; }
