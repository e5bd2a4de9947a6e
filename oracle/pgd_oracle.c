/*
 * Oracle for paged grouped-query decode attention with an optional per-head
 * sink logit and an optional sliding window.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, helper or table with the
 * CUDA library, and it is deliberately plain and slow: every quantity is a
 * double, every sum is a straight loop in the order the definition states.
 *
 * Sources (model-card pages of the "Nest" model zoo):
 *  - Mistral 7B Instruct v0.3, src/attention.linnet,
 *    GroupedQueryAttention.decode_paged: the new token's key and value are
 *    written at its place in the page pool (page_slots, write_tokens), then
 *    the row's queries attend over the row's pages up to and including its
 *    position, with scale rsqrt(head_dim).
 *  - Mistral 7B Instruct v0.3, README "Entries", decode_paged: the pool is
 *    one cache row of MaxSeq positions cut into pages of PageSize (64)
 *    positions, and row b's positions lie in the pages table[b] lists.
 *  - GPT-OSS 20B, README "Attention sinks" and src/attention.linnet header:
 *    one learned logit per query head joins the row of scores as an extra
 *    key, takes part in the softmax and is dropped, i.e. it enters only the
 *    denominator.
 *  - GPT-OSS 20B, src/attention.linnet, SinkAttention.decode_rows: key s is
 *    seen by the query at position n when s <= n and s > n - window.
 *  - GPT-OSS 20B, README (grouping of sink_attention): query heads are
 *    grouped by the key/value head they share, [B, KvHeads, G, Q, D], so
 *    query head h reads key/value head h / G.
 *  - Mistral 7B Instruct v0.3, src/attention.linnet, prefill_paged and the
 *    model's prefill_paged entry: packed prompt tokens are written at the
 *    caller's slots, and token p attends over its row's pages
 *    (table[rows[p]]) up to its position; GPT-OSS 20B, prefill_packed: the
 *    same window and sinks apply to prompt tokens.
 *
 * Readings where the pages leave a step open (each also listed in the
 * design notes):
 *  - page_slots(table, positions)[b] = table[b][n / P] * P + n % P, the
 *    position's index along the pool's MaxSeq axis (its body is not printed).
 *  - The sink is a logit in score space: it is not multiplied by the scale.
 *  - window <= 0 means no window (full causal attention).
 *  - A row with positions[b] < 0 is inactive: nothing is written for it and
 *    its output is zero (the pages compute such rows along and ignore them).
 *
 * Parity status: every function here is pinned by the CPU test suite against
 * closed forms, brute force with an explicit K+1 score column, a library
 * attention routine, and layout invariants.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ERANGE 2
#define ORC_ENOMEM 3

/* Pool layouts.  Both hold, for each (page, kv head), a contiguous tile of
 * page_size positions x head_dim values. */
#define ORC_PAGE_MAJOR 0 /* [num_pages][kv_heads][page_size][head_dim] */
#define ORC_HEAD_MAJOR 1 /* [kv_heads][num_pages * page_size][head_dim]  */

/* A bf16 value is the top half of an IEEE binary32; widening is exact. */
static double bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Element offset of (slot, kv head, dim) in a pool. */
static int64_t pool_offset(int layout, int64_t slot, int kv_head, int d, int kv_heads,
                           int head_dim, int page_size, int num_pages) {
  int64_t page = slot / page_size;
  int64_t in_page = slot % page_size;
  if (layout == ORC_PAGE_MAJOR)
    return ((page * kv_heads + kv_head) * page_size + in_page) * head_dim + d;
  return ((int64_t)kv_head * num_pages * page_size + slot) * head_dim + d;
}

/* page_slots: the pool position of each row's new token; -1 for an inactive
 * row.  Returns ORC_ERANGE if a position lies beyond the table's width or a
 * listed page lies outside the pool. */
int orc_page_slots(int rows, int max_pages, int page_size, int num_pages,
                   const int32_t* table, const int32_t* positions, int64_t* slots) {
  if (rows < 0 || max_pages <= 0 || page_size <= 0 || num_pages <= 0) return ORC_EINVAL;
  if (rows > 0 && (!table || !positions || !slots)) return ORC_EINVAL;
  for (int b = 0; b < rows; ++b) {
    int32_t n = positions[b];
    if (n < 0) {
      slots[b] = -1;
      continue;
    }
    int64_t page_index = n / page_size;
    if (page_index >= max_pages) return ORC_ERANGE;
    int32_t page = table[(int64_t)b * max_pages + page_index];
    if (page < 0 || page >= num_pages) return ORC_ERANGE;
    slots[b] = (int64_t)page * page_size + n % page_size;
  }
  return ORC_OK;
}

/* write_tokens: row b's new key (or value), kv_new[b][h][:], goes to slot
 * slots[b] of every kv head h of the pool.  Rows with slots[b] < 0 write
 * nothing. */
int orc_write_tokens(int rows, int kv_heads, int head_dim, int page_size, int num_pages,
                     int layout, const int64_t* slots, const uint16_t* kv_new,
                     uint16_t* pool) {
  if (rows < 0 || kv_heads <= 0 || head_dim <= 0 || page_size <= 0 || num_pages <= 0)
    return ORC_EINVAL;
  if (layout != ORC_PAGE_MAJOR && layout != ORC_HEAD_MAJOR) return ORC_EINVAL;
  for (int b = 0; b < rows; ++b) {
    if (slots[b] < 0) continue;
    if (slots[b] >= (int64_t)num_pages * page_size) return ORC_ERANGE;
    for (int h = 0; h < kv_heads; ++h)
      for (int d = 0; d < head_dim; ++d)
        pool[pool_offset(layout, slots[b], h, d, kv_heads, head_dim, page_size, num_pages)] =
            kv_new[((int64_t)b * kv_heads + h) * head_dim + d];
  }
  return ORC_OK;
}

/* Copies row b's positions 0..n out of the pool into a contiguous
 * [kv_heads][n + 1][head_dim] buffer, following table[b]. */
static int gather_row(int b, int n, int max_pages, int kv_heads, int head_dim, int page_size,
                      int num_pages, int layout, const int32_t* table, const uint16_t* pool,
                      uint16_t* dst) {
  for (int s = 0; s <= n; ++s) {
    int64_t page_index = s / page_size;
    if (page_index >= max_pages) return ORC_ERANGE;
    int32_t page = table[(int64_t)b * max_pages + page_index];
    if (page < 0 || page >= num_pages) return ORC_ERANGE;
    int64_t slot = (int64_t)page * page_size + s % page_size;
    for (int h = 0; h < kv_heads; ++h)
      for (int d = 0; d < head_dim; ++d)
        dst[((int64_t)h * (n + 1) + s) * head_dim + d] =
            pool[pool_offset(layout, slot, h, d, kv_heads, head_dim, page_size, num_pages)];
  }
  return ORC_OK;
}

/* One query head of one row.
 *   q      [head_dim]            the query
 *   k, v   [key_stride rows][head_dim]; keys 0..n are the row's positions
 *   sink   the head's sink logit, or -INFINITY for none
 * Attended set A = { s : 0 <= s <= n, and window <= 0 or s > n - window }.
 * Scores s_j = scale * sum_d q[d] k[j][d].  With m = max(max_j s_j, sink)
 * and Z = sum_j exp(s_j - m) + exp(sink - m), out = sum_j exp(s_j - m) v[j] / Z.
 * lse = m + log Z includes the sink; lse_real is the log-sum-exp of the real
 * scores alone. */
static int attend_head(const uint16_t* q, const uint16_t* k, const uint16_t* v, int n,
                       int head_dim, int window, double scale, double sink, double* out,
                       double* lse, double* lse_real) {
  int lo = 0;
  if (window > 0 && n - window + 1 > 0) lo = n - window + 1;
  int count = n - lo + 1;
  double* score = (double*)malloc(sizeof(double) * (size_t)count);
  if (!score) return ORC_ENOMEM;

  double m_real = -INFINITY;
  for (int j = 0; j < count; ++j) {
    const uint16_t* kj = k + (int64_t)(lo + j) * head_dim;
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d) dot += bf16_value(q[d]) * bf16_value(kj[d]);
    score[j] = scale * dot;
    if (score[j] > m_real) m_real = score[j];
  }
  double m = m_real > sink ? m_real : sink;

  double z = (sink == -INFINITY) ? 0.0 : exp(sink - m);
  double z_real = 0.0;
  for (int j = 0; j < count; ++j) {
    z += exp(score[j] - m);
    z_real += exp(score[j] - m_real);
  }
  for (int d = 0; d < head_dim; ++d) out[d] = 0.0;
  for (int j = 0; j < count; ++j) {
    double p = exp(score[j] - m) / z;
    const uint16_t* vj = v + (int64_t)(lo + j) * head_dim;
    for (int d = 0; d < head_dim; ++d) out[d] += p * bf16_value(vj[d]);
  }
  *lse = m + log(z);
  *lse_real = m_real + log(z_real);
  free(score);
  return ORC_OK;
}

/* Shared argument block for the per-row workers. */
typedef struct {
  int rows, q_heads, kv_heads, head_dim, window;
  double scale;
  const uint16_t* q;
  const int32_t* positions;
  const float* sinks;
  double *out, *lse, *lse_real;
  /* contiguous source */
  int key_stride;
  const uint16_t *k, *v;
  /* paged source */
  int paged, max_pages, page_size, num_pages, layout;
  const int32_t* table;
  /* prefill: token b reads table row row_of[b] (of table_rows); NULL: row b */
  const int32_t* row_of;
  int table_rows;
  const uint16_t *k_pool, *v_pool;
  /* work distribution */
  int nthreads, thread;
  int status;
} job_t;

static int run_row(job_t* job, int b) {
  int group = job->q_heads / job->kv_heads;
  int d_head = job->head_dim;
  int n = job->positions[b];
  if (n < 0) {
    for (int h = 0; h < job->q_heads; ++h) {
      for (int d = 0; d < d_head; ++d) job->out[((int64_t)b * job->q_heads + h) * d_head + d] = 0.0;
      job->lse[(int64_t)b * job->q_heads + h] = -INFINITY;
      job->lse_real[(int64_t)b * job->q_heads + h] = -INFINITY;
    }
    return ORC_OK;
  }
  const uint16_t *k_rows, *v_rows;
  uint16_t *k_buf = NULL, *v_buf = NULL;
  int64_t stride;
  if (job->paged) {
    int trow = b;
    if (job->row_of) {
      trow = job->row_of[b];
      if (trow < 0 || trow >= job->table_rows) return ORC_ERANGE;
    }
    size_t count = (size_t)job->kv_heads * (size_t)(n + 1) * (size_t)d_head;
    k_buf = (uint16_t*)malloc(count * sizeof(uint16_t));
    v_buf = (uint16_t*)malloc(count * sizeof(uint16_t));
    if (!k_buf || !v_buf) {
      free(k_buf);
      free(v_buf);
      return ORC_ENOMEM;
    }
    int rc = gather_row(trow, n, job->max_pages, job->kv_heads, d_head, job->page_size,
                        job->num_pages, job->layout, job->table, job->k_pool, k_buf);
    if (rc == ORC_OK)
      rc = gather_row(trow, n, job->max_pages, job->kv_heads, d_head, job->page_size,
                      job->num_pages, job->layout, job->table, job->v_pool, v_buf);
    if (rc != ORC_OK) {
      free(k_buf);
      free(v_buf);
      return rc;
    }
    k_rows = k_buf;
    v_rows = v_buf;
    stride = n + 1;
  } else {
    if (n >= job->key_stride) return ORC_ERANGE;
    k_rows = job->k + (int64_t)b * job->kv_heads * job->key_stride * d_head;
    v_rows = job->v + (int64_t)b * job->kv_heads * job->key_stride * d_head;
    stride = job->key_stride;
  }
  int rc = ORC_OK;
  for (int h = 0; h < job->q_heads && rc == ORC_OK; ++h) {
    int g = h / group;
    double sink = job->sinks ? (double)job->sinks[h] : -INFINITY;
    int64_t bh = (int64_t)b * job->q_heads + h;
    rc = attend_head(job->q + bh * d_head, k_rows + (int64_t)g * stride * d_head,
                     v_rows + (int64_t)g * stride * d_head, n, d_head, job->window, job->scale,
                     sink, job->out + bh * d_head, job->lse + bh, job->lse_real + bh);
  }
  free(k_buf);
  free(v_buf);
  return rc;
}

static void* run_rows(void* arg) {
  job_t* job = (job_t*)arg;
  job->status = ORC_OK;
  for (int b = job->thread; b < job->rows; b += job->nthreads) {
    int rc = run_row(job, b);
    if (rc != ORC_OK) {
      job->status = rc;
      break;
    }
  }
  return NULL;
}

static int run_job(job_t* base, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > base->rows && base->rows > 0) nthreads = base->rows;
  if (nthreads <= 1) {
    base->nthreads = 1;
    base->thread = 0;
    run_rows(base);
    return base->status;
  }
  job_t* jobs = (job_t*)malloc(sizeof(job_t) * (size_t)nthreads);
  pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!jobs || !tids) {
    free(jobs);
    free(tids);
    return ORC_ENOMEM;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *base;
    jobs[t].nthreads = nthreads;
    jobs[t].thread = t;
    if (pthread_create(&tids[t], NULL, run_rows, &jobs[t]) != 0) break;
    ++started;
  }
  int rc = started == nthreads ? ORC_OK : ORC_ENOMEM;
  for (int t = 0; t < started; ++t) {
    pthread_join(tids[t], NULL);
    if (jobs[t].status != ORC_OK) rc = jobs[t].status;
  }
  free(jobs);
  free(tids);
  return rc;
}

static int check_heads(int rows, int q_heads, int kv_heads, int head_dim) {
  if (rows < 0 || q_heads <= 0 || kv_heads <= 0 || head_dim <= 0) return ORC_EINVAL;
  if (q_heads % kv_heads != 0) return ORC_EINVAL;
  return ORC_OK;
}

/* Decode attention over contiguous per-row caches (the decode_rows layout):
 *   q        [rows][q_heads][head_dim]              bf16 bits
 *   k, v     [rows][kv_heads][key_stride][head_dim]  bf16 bits
 *   positions[rows]  int32; row b attends over keys 0..positions[b]
 *   sinks    [q_heads] float or NULL
 *   out      [rows][q_heads][head_dim] double; lse, lse_real [rows][q_heads]. */
int orc_decode_rows(int rows, int q_heads, int kv_heads, int head_dim, int key_stride,
                    const uint16_t* q, const uint16_t* k, const uint16_t* v,
                    const int32_t* positions, const float* sinks, int window, float scale,
                    double* out, double* lse, double* lse_real, int nthreads) {
  int rc = check_heads(rows, q_heads, kv_heads, head_dim);
  if (rc != ORC_OK) return rc;
  if (key_stride <= 0) return ORC_EINVAL;
  job_t job;
  memset(&job, 0, sizeof job);
  job.rows = rows;
  job.q_heads = q_heads;
  job.kv_heads = kv_heads;
  job.head_dim = head_dim;
  job.window = window;
  job.scale = (double)scale;
  job.q = q;
  job.positions = positions;
  job.sinks = sinks;
  job.out = out;
  job.lse = lse;
  job.lse_real = lse_real;
  job.key_stride = key_stride;
  job.k = k;
  job.v = v;
  return run_job(&job, nthreads);
}

/* Decode attention over a page pool: row b's keys 0..positions[b] are found
 * through table[b] (max_pages entries per row), gathered, and attended to
 * exactly as orc_decode_rows does. */
int orc_decode_paged(int rows, int q_heads, int kv_heads, int head_dim, int page_size,
                     int num_pages, int max_pages, int layout, const uint16_t* q,
                     const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* table,
                     const int32_t* positions, const float* sinks, int window, float scale,
                     double* out, double* lse, double* lse_real, int nthreads) {
  int rc = check_heads(rows, q_heads, kv_heads, head_dim);
  if (rc != ORC_OK) return rc;
  if (page_size <= 0 || num_pages <= 0 || max_pages <= 0) return ORC_EINVAL;
  if (layout != ORC_PAGE_MAJOR && layout != ORC_HEAD_MAJOR) return ORC_EINVAL;
  job_t job;
  memset(&job, 0, sizeof job);
  job.rows = rows;
  job.q_heads = q_heads;
  job.kv_heads = kv_heads;
  job.head_dim = head_dim;
  job.window = window;
  job.scale = (double)scale;
  job.q = q;
  job.positions = positions;
  job.sinks = sinks;
  job.out = out;
  job.lse = lse;
  job.lse_real = lse_real;
  job.paged = 1;
  job.max_pages = max_pages;
  job.page_size = page_size;
  job.num_pages = num_pages;
  job.layout = layout;
  job.table = table;
  job.k_pool = k_pool;
  job.v_pool = v_pool;
  return run_job(&job, nthreads);
}

/* Paged prefill (prefill_paged / paged_prefill_attention): P packed tokens;
 * token p is position positions[p] of the request in table row rows[p]
 * (table has table_rows rows of max_pages entries).  Its key and value were
 * written at its slot beforehand (orc_write_tokens with the caller's
 * slots), and its query attends over its row's pages up to and including
 * its own position, within the window, with the sink in the denominator:
 * exactly a decode step of row rows[p] at position positions[p].
 *   q [P][q_heads][head_dim] bf16; out [P][q_heads][head_dim] double. */
int orc_prefill_paged(int tokens, int q_heads, int kv_heads, int head_dim, int page_size,
                      int num_pages, int table_rows, int max_pages, int layout,
                      const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                      const int32_t* table, const int32_t* rows, const int32_t* positions,
                      const float* sinks, int window, float scale, double* out, double* lse,
                      double* lse_real, int nthreads) {
  int rc = check_heads(tokens, q_heads, kv_heads, head_dim);
  if (rc != ORC_OK) return rc;
  if (page_size <= 0 || num_pages <= 0 || max_pages <= 0 || table_rows <= 0 || !rows)
    return ORC_EINVAL;
  if (layout != ORC_PAGE_MAJOR && layout != ORC_HEAD_MAJOR) return ORC_EINVAL;
  job_t job;
  memset(&job, 0, sizeof job);
  job.rows = tokens;
  job.q_heads = q_heads;
  job.kv_heads = kv_heads;
  job.head_dim = head_dim;
  job.window = window;
  job.scale = (double)scale;
  job.q = q;
  job.positions = positions;
  job.sinks = sinks;
  job.out = out;
  job.lse = lse;
  job.lse_real = lse_real;
  job.paged = 1;
  job.max_pages = max_pages;
  job.page_size = page_size;
  job.num_pages = num_pages;
  job.layout = layout;
  job.table = table;
  job.k_pool = k_pool;
  job.v_pool = v_pool;
  job.row_of = rows;
  job.table_rows = table_rows;
  return run_job(&job, nthreads);
}

/* ------------------------------------------------------------------------
 * Rotary position embedding (Mistral 7B Instruct v0.3 model files,
 * src/rope.linnet, `tables`; applied by rope_rows in decode_paged).
 *
 * The tables are computed in f32 as the pages write them,
 *   inv_freq[i] = exp(-(i * 2 / D) * log(theta)),  angle = pos * inv_freq[i],
 * and cos/sin of the angle are cast to the model dtype (bf16), each
 * frequency repeated over both halves of the head dimension; so dimension i
 * pairs with i + D/2 (the rotate-half form; the GPT-OSS rope page notes the
 * half-split and repeated-table forms compute the same rotation):
 *   out[i]       = x[i] cos_i - x[i + D/2] sin_i
 *   out[i + D/2] = x[i + D/2] cos_i + x[i] sin_i
 * Reading where the pages leave it open: the rotation itself is exact (fp64
 * here) and its result is rounded once to bf16. */

/* Round-to-nearest-even from binary32 to bf16 (the top 16 bits), from the
 * IEEE definition: add half an ulp of the result, plus one if the kept part
 * is odd, then truncate; NaNs stay NaNs. */
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x40u);
  uint32_t keep_odd = (u >> 16) & 1u;
  u += 0x7fffu + keep_odd;
  return (uint16_t)(u >> 16);
}

static uint16_t f64_to_bf16_rne(double x) {
  /* Through binary32 first is exact enough: a double rounding can only
   * matter at a bf16 tie, which the 16 extra bits of binary32 make
   * vanishingly rare; the tests compare the final values within one ulp. */
  return f32_to_bf16_rne((float)x);
}

/* cos/sin table entries (bf16 bit patterns) of position pos for i < D/2. */
int orc_rope_table(int head_dim, float theta, int pos, uint16_t* cos_out, uint16_t* sin_out) {
  if (head_dim <= 0 || head_dim % 2 || pos < 0) return ORC_EINVAL;
  const float log_theta = logf(theta);
  for (int i = 0; i < head_dim / 2; ++i) {
    const float scaled = ((float)i * 2.0f) / (float)head_dim;
    const float inv_freq = expf(-scaled * log_theta);
    const float angle = (float)pos * inv_freq;
    cos_out[i] = f64_to_bf16_rne(cos((double)angle));
    sin_out[i] = f64_to_bf16_rne(sin((double)angle));
  }
  return ORC_OK;
}

/* rope_rows: x [n][heads][head_dim] (bf16 bits) rotated at positions[r];
 * rows with a negative position are copied unchanged. */
int orc_rope(int n, int heads, int head_dim, float theta, const uint16_t* x,
             const int32_t* positions, uint16_t* out) {
  if (n < 0 || heads <= 0 || head_dim <= 0 || head_dim % 2) return ORC_EINVAL;
  const int half = head_dim / 2;
  uint16_t* c = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)half);
  uint16_t* s = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)half);
  if (!c || !s) {
    free(c);
    free(s);
    return ORC_ENOMEM;
  }
  int rc = ORC_OK;
  for (int r = 0; r < n && rc == ORC_OK; ++r) {
    const uint16_t* xr = x + (int64_t)r * heads * head_dim;
    uint16_t* orow = out + (int64_t)r * heads * head_dim;
    if (positions[r] < 0) {
      memcpy(orow, xr, sizeof(uint16_t) * (size_t)heads * head_dim);
      continue;
    }
    rc = orc_rope_table(head_dim, theta, positions[r], c, s);
    for (int h = 0; h < heads && rc == ORC_OK; ++h)
      for (int i = 0; i < half; ++i) {
        const double a = bf16_value(xr[h * head_dim + i]);
        const double b = bf16_value(xr[h * head_dim + i + half]);
        const double ci = bf16_value(c[i]), si = bf16_value(s[i]);
        orow[h * head_dim + i] = f64_to_bf16_rne(a * ci - b * si);
        orow[h * head_dim + i + half] = f64_to_bf16_rne(b * ci + a * si);
      }
  }
  free(c);
  free(s);
  return rc;
}
