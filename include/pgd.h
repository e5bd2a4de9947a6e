/*
 * pgd.h -- C ABI of libpgd: paged grouped-query decode attention for GB300
 * (sm_103a), with an optional per-head attention-sink logit and an optional
 * sliding window.
 *
 * One serving step of a continuous batch: every row b has one new token at
 * position positions[b].  Its key and value are appended to a pool of
 * 64-position pages at the place the row's page table gives, then the row's
 * query heads attend over the row's pages up to and including that position.
 *
 * Operation definitions (model-card pages of the "Nest" zoo):
 *   - Mistral 7B Instruct v0.3, src/attention.linnet,
 *     GroupedQueryAttention.decode_paged, and README "Entries" (decode_paged):
 *     page_slots(table, positions), write_tokens into the pool, then
 *     paged_attention(q, cache_k, cache_v, table, positions, rsqrt(head_dim))
 *     (pgd_kv_append_paged + pgd_paged_decode_attention, or both in one
 *     launch: pgd_paged_decode_step).
 *   - GPT-OSS 20B, README "Attention sinks": one learned logit per query head
 *     joins the scores as an extra key and is dropped after the softmax, so it
 *     adds exp(sink - m) to the softmax denominator only.
 *   - GPT-OSS 20B, src/attention.linnet, SinkAttention.decode_rows: key s is
 *     seen by the query at position n when s <= n and s > n - window.
 *   - GPT-OSS 20B, README (grouped sink_attention): query head h reads kv head
 *     h / (num_q_heads / num_kv_heads); K/V are never copied per query head.
 *
 * Conventions for every entry point:
 *   - All pointers except `dims`, `opts`, the `count` of
 *     pgd_attention_kernel_count and the result of pgd_status_string are
 *     DEVICE pointers owned by the caller.  The library
 *     allocates no memory; scratch is the caller's `workspace`.
 *   - bf16 tensors are passed as raw 16-bit storage.  Every bf16 pointer and
 *     the workspace must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Arguments are validated on the host before anything
 *     is launched; a non-zero return means nothing was enqueued.
 *   - Row b is inactive when positions[b] < 0: nothing is appended for it and
 *     its output is zero.
 *   - Bad table entries or positions found on the device do not fault: the
 *     affected row is skipped (its output zero) and a sticky device error
 *     word is set, which pgd_get_device_error reads and clears.
 */
#ifndef PGD_H_
#define PGD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PGD_API __attribute__((visibility("default")))
#else
#define PGD_API
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st* pgd_stream_t;

/* Status codes. */
enum {
  PGD_OK = 0,
  PGD_EINVAL = 1,          /* NULL pointer, bad shape, misaligned pointer */
  PGD_EUNSUPPORTED = 2,    /* head_dim not 64/128, page_size not 64, group > 8 */
  PGD_ECUDA = 3,           /* a CUDA runtime or driver call failed */
  PGD_EDEVICE_BOUNDS = 4,  /* device: table entry or position out of range */
  PGD_EDEVICE_TIMEOUT = 5, /* device: a pipeline wait gave up (bounded waits) */
  PGD_EWORKSPACE = 6,      /* workspace smaller than pgd_paged_decode_workspace_bytes */
  PGD_ESCRATCH_LIMIT = 7   /* problem needs more scratch than PGD_STATIC_SCRATCH_BYTES */
};

/* Pool layouts.  In both, the 64 x head_dim values of one (page, kv head)
 * form one contiguous tile, so a page tile is read with a single copy. */
enum {
  PGD_PAGE_MAJOR = 0, /* [num_pages][num_kv_heads][64][head_dim] */
  PGD_HEAD_MAJOR = 1, /* [num_kv_heads][num_pages * 64][head_dim]: the pages'
                         own cache_k[0] layout, [KvHeads, MaxSeq, D] */
  PGD_ROW_MAJOR = 2   /* [num_pages / P][num_kv_heads][P * 64][head_dim] with
                         P = max_pages_per_row: the dense per-row caches of
                         decode_rows, [Batch, KvHeads, MaxSeq, D] with
                         MaxSeq = 64 P (GPT-OSS 20B and Mistral 7B Instruct
                         v0.3 model files, src/attention.linnet, cache_k and
                         decode_rows); page b * P + j is positions
                         64 j .. 64 j + 63 of row b.  With this layout the
                         table may be NULL: row b's pages are then
                         b * P + j (decode_rows), and rows <= num_pages / P. */
};

typedef struct {
  int32_t rows;              /* R >= 0 rows of the continuous batch */
  int32_t num_q_heads;       /* Hq > 0 */
  int32_t num_kv_heads;      /* Hkv > 0, Hq % Hkv == 0, Hq / Hkv <= 8 */
  int32_t head_dim;          /* D: 64 or 128 */
  int32_t page_size;         /* positions per page: must be 64 */
  int32_t num_pages;         /* pool capacity in pages, >= 1 */
  int32_t max_pages_per_row; /* table row stride (entries per row), >= 1 */
  int32_t layout;            /* PGD_PAGE_MAJOR, PGD_HEAD_MAJOR or PGD_ROW_MAJOR */
} pgd_dims;

/* Kernel variants.  All compute the same function; they differ in where the
 * per-page Q.K^T and P.V products run and in how tokens share page loads. */
enum {
  PGD_KERNEL_AUTO = 0,          /* decode: windows of 1..128 positions go to the
                                   window kernel (the warps given each row and
                                   kv head copy exactly the window's K/V rows;
                                   mma.sync products; no splits), and so does
                                   full attention over a table of at most 10
                                   pages (head_dim 64) or 4 (128) when the
                                   rows x kv heads are between half and all of
                                   the device's SMs and opts->pages_per_split
                                   is 0 (the whole table its window); anything
                                   else to TENSOR_CORE; prefill: when the tokens average
                                   at least 8 per table row (prompt chunks),
                                   PREFILL_UMMA, whose blocks x kv heads, when
                                   at most half the device's SMs, are cut into
                                   key parts (see pgd_paged_prefill_attention)
                                   or, where too short to cut, at head_dim 128
                                   go to PREFILL_PAIR; otherwise as decode,
                                   per token */
  PGD_KERNEL_TENSOR_CORE = 1,   /* mma.sync bf16 products, fp32 accumulate, per token,
                                   key range split over CTAs + combine */
  PGD_KERNEL_CUDA_CORE = 2,     /* fp32 FMA products on the CUDA cores, per token */
  PGD_KERNEL_PREFILL_TILED = 3, /* prefill only: blocks of tokens share each page
                                   load (mma.sync tensor cores, no key splits) */
  PGD_KERNEL_PREFILL_UMMA = 4,  /* prefill only: persistent, two tiles of 128
                                   query rows per block on the tcgen05 tensor
                                   cores (TMEM accumulators), no key splits
                                   when named (AUTO may add key parts); uses
                                   the start of the workspace for its work
                                   counter and block order */
  PGD_KERNEL_PREFILL_PAIR = 5   /* prefill only, head_dim 128: the same blocks
                                   on pairs of SMs (clusters of two CTAs, one
                                   query tile each, sharing every tcgen05
                                   product; each CTA loads every other page,
                                   so one product spans 128 keys); the same
                                   use of the workspace */
};

/* Optional tuning of the decode launch; pass NULL for the defaults.  The same
 * options must be passed to pgd_paged_decode_workspace_bytes and to
 * pgd_paged_decode_attention. */
typedef struct {
  int32_t pages_per_split; /* pages one CTA streams; 0 = chosen from dims and
                              the device's SM count */
  int32_t kernel;          /* PGD_KERNEL_*; 0 = auto */
} pgd_decode_options;

/*
 * kv_append_paged -- page_slots + write_tokens.
 *   k_new, v_new  bf16 [R][Hkv][D]: the new token's key and value per row.
 *   table         int32 [R][max_pages_per_row]: row b's pages in order
 *                 (NULL with PGD_ROW_MAJOR: row b's pages are b * P + j, i.e.
 *                 write_rows into dense per-row caches).
 *   positions     int32 [R]: the new token's 0-based position (< 0: inactive).
 *   k_pool,v_pool bf16 pools in dims->layout, num_pages pages each.
 * Row b's token is written at position positions[b] % 64 of page
 * table[b][positions[b] / 64], for every kv head.  Two active rows must not
 * name the same slot (the result would be either row's value).
 * Device errors: positions[b] / 64 >= max_pages_per_row, or a table entry
 * outside [0, num_pages): nothing is written for that row and
 * PGD_EDEVICE_BOUNDS is recorded.
 */
PGD_API int pgd_kv_append_paged(const pgd_dims* dims, const void* k_new, const void* v_new,
                        const int32_t* table, const int32_t* positions, void* k_pool,
                        void* v_pool, pgd_stream_t stream);

/*
 * page_slots -- the pool position of each token (Mistral 7B Instruct v0.3
 * model files, src/attention.linnet, decode_paged: page_slots(table,
 * positions); README "Entries": row b's positions lie in the pages table[b]
 * lists): slots[p] = table[r][n / 64] * 64 + n % 64 with n = positions[p]
 * and r = rows[p] (rows NULL: r = p).  n < 0 gives -1.
 *   dims->rows   number of tokens P; dims->max_pages_per_row the table width.
 *   table_rows   rows of `table` (ignored when rows is NULL: P rows).
 * Device errors: n / 64 beyond the table, r outside the table, or a listed
 * page outside the pool -> slots[p] = -1 and PGD_EDEVICE_BOUNDS recorded.
 */
PGD_API int pgd_page_slots(const pgd_dims* dims, int32_t table_rows, const int32_t* table,
                           const int32_t* rows, const int32_t* positions, int32_t* slots,
                           pgd_stream_t stream);

/*
 * kv_write_slots -- prefill's write_tokens at caller-given places (Mistral 7B
 * Instruct v0.3 model files, src/attention.linnet, prefill_paged: each
 * packed prompt token is written at its place in the pool, `slots`).
 *   dims->rows    P tokens; dims->max_pages_per_row is not used.
 *   k_new, v_new  bf16 [P][Hkv][D].
 *   slots         int32 [P]: pool position slot = page * 64 + offset, the
 *                 same numbering page_slots produces; < 0: padding, skipped.
 * Device errors: slot / 64 >= num_pages -> nothing written for that token,
 * PGD_EDEVICE_BOUNDS recorded.
 */
PGD_API int pgd_kv_write_slots(const pgd_dims* dims, const void* k_new, const void* v_new,
                               const int32_t* slots, void* k_pool, void* v_pool,
                               pgd_stream_t stream);

/*
 * rope_append_paged -- rope_rows + append in one launch (Mistral 7B Instruct
 * v0.3 model files, src/attention.linnet, decode_paged: q and k rotated at
 * positions[b], then write_tokens; src/rope.linnet, tables with base theta).
 *   theta         rotary base (1e6 for Mistral v0.3 and Qwen2.5).
 *   q             bf16 [R][Hq][D], rotated in place (NULL: k only).
 *   k_new, v_new  bf16 [R][Hkv][D], un-rotated; k is rotated on its way into
 *                 the pool, v copied.
 *   table, positions, pools  as for pgd_kv_append_paged; or
 *   slots         int32 [R]: explicit pool positions (prefill), overriding
 *                 the table (which may then be NULL); NULL otherwise.
 * Tables as the pages compute them: inv_freq[i] = exp(-(2i / D) log theta)
 * and angle = position * inv_freq[i] in f32, cos/sin rounded to bf16; dims i
 * and i + D/2 are rotated together and each result rounded to bf16.
 * Rows with positions[b] < 0 are left alone.  Device errors as for
 * pgd_kv_append_paged (the row is then left alone, q included).
 */
PGD_API int pgd_rope_append_paged(const pgd_dims* dims, float theta, void* q,
                                  const void* k_new, const void* v_new, const int32_t* table,
                                  const int32_t* positions, const int32_t* slots, void* k_pool,
                                  void* v_pool, pgd_stream_t stream);

/*
 * Bytes of device workspace pgd_paged_decode_attention needs for these dims
 * and options on the current device: split partials (m, l and an unnormalised
 * fp32 accumulator per row, query head and split), with room as well for the
 * key parts a prefill call of these dims may be cut into (one more split's
 * worth than their number).  0 if dims are invalid.
 */
PGD_API size_t pgd_paged_decode_workspace_bytes(const pgd_dims* dims, const pgd_decode_options* opts);

/*
 * attention_kernel_count -- how many kernels one attention call with these
 * arguments launches on the current device (for callers that count launches
 * or size CUDA graphs; the pages have no counterpart).
 *   table_rows  0 for pgd_paged_decode_attention; the table_rows argument of
 *               pgd_paged_prefill_attention (> 0) for a prefill call.
 *   window, opts  as passed to that call.
 *   count       out: 0 when dims->rows == 0; 1 for AUTO with a window of
 *               1..128 positions or on a table the window kernel takes
 *               whole (see PGD_KERNEL_AUTO); for PREFILL_UMMA and
 *               PREFILL_PAIR 2 without a
 *               window when the tokens form at most 4096 blocks of
 *               2 x (128 / group) (a pass that orders the blocks longest
 *               first, then the prefill kernel), else 1 (the kernel, after
 *               one 4-byte cudaMemsetAsync), plus 1 (the combine) when AUTO
 *               cuts the blocks into key parts; 1 for PREFILL_TILED and for
 *               split kernels whose rows all fit one split (it writes every
 *               output); 2 when a row can span several splits (split kernel
 *               + combine kernel).
 * Returns PGD_EINVAL for a NULL count, negative table_rows or a kernel the
 * call would reject, and the pgd_dims checks' codes.
 */
PGD_API int pgd_attention_kernel_count(const pgd_dims* dims, int32_t table_rows, int32_t window,
                                       const pgd_decode_options* opts, int32_t* count);

/*
 * paged_decode_attention -- paged_attention with an optional sink and window.
 *   q          bf16 [R][Hq][D]: queries (rope already applied).
 *   k_pool, v_pool  the pools, holding each active row's positions
 *              0..positions[b] (append first: the new token attends to itself).
 *   table, positions  as for pgd_kv_append_paged (the table may be NULL with
 *              PGD_ROW_MAJOR: decode_rows over dense per-row caches).
 *   sinks      fp32 [Hq] sink logits (score space: not multiplied by scale),
 *              or NULL for none.
 *   window     > 0: row b attends to positions (n - window, n];
 *              <= 0: full causal attention over 0..n.
 *   scale      score scale, normally 1 / sqrt(D).
 *   out        bf16 [R][Hq][D], rounded to nearest even from fp32.
 *   workspace  >= pgd_paged_decode_workspace_bytes(dims, opts) bytes.
 * Query head h of row b uses kv head h / (Hq / Hkv).  For each row and head,
 * m = max(max_j s_j, sink), out = sum_j e^(s_j - m) v_j /
 * (sum_j e^(s_j - m) + e^(sink - m)) with s_j = scale * q . k_j, in fp32.
 * Device errors: as for pgd_kv_append_paged (for any attended page), plus
 * PGD_EDEVICE_TIMEOUT if a pipeline wait exceeded its limit; the output of
 * every (row, kv head group) whose pages were skipped, or whose split gave
 * up waiting, is zero.
 */
PGD_API int pgd_paged_decode_attention(const pgd_dims* dims, const void* q, const void* k_pool,
                               const void* v_pool, const int32_t* table,
                               const int32_t* positions, const float* sinks, int32_t window,
                               float scale, void* out, void* workspace, size_t workspace_bytes,
                               const pgd_decode_options* opts, pgd_stream_t stream);

/*
 * paged_decode_step -- pgd_kv_append_paged then pgd_paged_decode_attention
 * in one launch (plus the combine kernel when a row spans several splits):
 * the decode_paged step of the pages (Mistral 7B Instruct v0.3 model files,
 * src/attention.linnet, GroupedQueryAttention.decode_paged: write_tokens,
 * then paged_attention).  For each active row, the CTA that streams the
 * row's last page (per kv head) first writes k_new and v_new at the slot of
 * positions[b] and then loads that page, so the new token attends to itself.
 *   k_new, v_new  bf16 [R][Hkv][D]; k_pool, v_pool written as by
 *                 pgd_kv_append_paged.  Other arguments, the workspace and
 *                 the result as for pgd_paged_decode_attention.
 * Device errors as for pgd_paged_decode_attention; a row whose last split
 * reads a table entry outside the pool gets no append.
 */
PGD_API int pgd_paged_decode_step(const pgd_dims* dims, const void* q, const void* k_new,
                                  const void* v_new, void* k_pool, void* v_pool,
                                  const int32_t* table, const int32_t* positions,
                                  const float* sinks, int32_t window, float scale, void* out,
                                  void* workspace, size_t workspace_bytes,
                                  const pgd_decode_options* opts, pgd_stream_t stream);

/*
 * paged_prefill_attention -- packed prompt tokens over their rows' pages
 * (Mistral 7B Instruct v0.3 model files, src/attention.linnet,
 * prefill_paged / step_paged and the model's prefill_paged entry; window and
 * sinks as GPT-OSS 20B prefill_packed).  Token p is position positions[p]
 * of the request in table row rows[p]; its query attends over that row's
 * pages up to and including positions[p], within the window, with the sink
 * in the denominator -- the same function as a decode step of that row.
 * Write the tokens' keys and values first (pgd_kv_write_slots).
 *   dims->rows    P tokens; dims->max_pages_per_row is the table width.
 *   table_rows    rows of `table` (int32 [table_rows][max_pages_per_row]).
 *   q, out        bf16 [P][Hq][D]; rows, positions int32 [P].
 *   Others as for pgd_paged_decode_attention; the workspace size is
 *   pgd_paged_decode_workspace_bytes(dims, opts) with dims->rows = P.
 * step_paged (prompts and one decode step per row in one pass) is one call
 * over the concatenation: the step of row b is a token with rows = b at its
 * step position.
 * Kernels (opts->kernel): AUTO chooses PREFILL_UMMA (tokens in blocks of
 * 2 x 128 / (Hq / Hkv), two query tiles, share every page load; persistent,
 * one CTA per SM; each item's Q copied in with TMA; without a window the
 * blocks are taken longest first) when P >= 8 * table_rows, else the
 * per-token decode kernels (the window kernel for windows of 1..128
 * positions, the TENSOR_CORE split kernel otherwise).  When the blocks x
 * Hkv (the work items) are at most half the device's SM count, AUTO cuts
 * each item's pages into key parts -- min(8, SMs / items, L / 8) of them,
 * L the table width in pages (with a window, the pages a block's keys can
 * span), if that is 2 or more -- each a work unit of its own that writes
 * partials (m, l and an unnormalised fp32 accumulator per token, head and
 * part) into the workspace, which a combine launch merges with the sink;
 * the results then differ from PREFILL_UMMA's by rounding only.  Where the
 * items are too short to cut, at head_dim 128 such calls go to
 * PREFILL_PAIR (the same blocks, two SMs each).
 * Device errors: rows[p] outside [0, table_rows), plus those of
 * pgd_paged_decode_attention; the token's output is zero.  After
 * PGD_EDEVICE_TIMEOUT (a pipeline wait gave up) the outputs of the tokens
 * whose work was abandoned are unspecified: the PREFILL_TILED,
 * PREFILL_UMMA and PREFILL_PAIR kernels stop without writing them.
 */
PGD_API int pgd_paged_prefill_attention(const pgd_dims* dims, int32_t table_rows, const void* q,
                                        const void* k_pool, const void* v_pool,
                                        const int32_t* table, const int32_t* rows,
                                        const int32_t* positions, const float* sinks,
                                        int32_t window, float scale, void* out, void* workspace,
                                        size_t workspace_bytes, const pgd_decode_options* opts,
                                        pgd_stream_t stream);

/*
 * paged_prefill_step -- the prefill call with the tokens' writes in it
 * (Mistral 7B Instruct v0.3 model files, src/attention.linnet, prefill_paged:
 * page_slots and write_tokens for every packed token, then the attention):
 * the same as pgd_page_slots + pgd_kv_write_slots + pgd_paged_prefill_attention
 * with the same arguments, in fewer launches.  Token p's k_new / v_new rows go
 * to position positions[p] % 64 of page table[rows[p]][positions[p] / 64]
 * (tokens with a negative position are not written), then every token
 * attends as in pgd_paged_prefill_attention, its own and its row's other new
 * keys included.
 *   k_new, v_new  bf16 [P][Hkv][D] device pointers, 16-byte aligned.
 *   k_pool, v_pool  written (the tokens' slots) and read.
 *   Others as for pgd_paged_prefill_attention.
 * Launches: one kernel writes the tokens (with PREFILL_UMMA or PREFILL_PAIR
 * its first CTA also prepares the attention kernel's work counter and block
 * order in the workspace), then the attention kernels; pgd_prefill_step_kernel_count
 * gives the number.  Two tokens with the same slot race, as with
 * pgd_kv_write_slots.
 * Device errors: a token whose row, page index or page is out of range is
 * reported (PGD_EDEVICE_BOUNDS), not written, and its output is zero; others
 * as for pgd_paged_prefill_attention.
 */
PGD_API int pgd_paged_prefill_step(const pgd_dims* dims, int32_t table_rows, const void* q,
                                   const void* k_new, const void* v_new, void* k_pool,
                                   void* v_pool, const int32_t* table, const int32_t* rows,
                                   const int32_t* positions, const float* sinks, int32_t window,
                                   float scale, void* out, void* workspace,
                                   size_t workspace_bytes, const pgd_decode_options* opts,
                                   pgd_stream_t stream);

/* Kernels one pgd_paged_prefill_step call with these arguments launches on
 * the current device: the write launch plus the attention kernels (for
 * PREFILL_UMMA and PREFILL_PAIR the attention kernel alone, its counter and
 * order prepared by the write launch, and the combine with key parts).  table_rows > 0; count 0 when dims->rows == 0.  Returns
 * PGD_EINVAL for a NULL count or table_rows <= 0, else as
 * pgd_attention_kernel_count. */
PGD_API int pgd_prefill_step_kernel_count(const pgd_dims* dims, int32_t table_rows,
                                          int32_t window, const pgd_decode_options* opts,
                                          int32_t* count);

/* Size of the library's own device scratch buffer used by
 * pgd_paged_decode_attention_static: 64 MiB on every device that loads the
 * library, held until the process exits. */
#define PGD_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * paged_decode_attention_static -- pgd_paged_decode_attention for callers that
 * cannot allocate device memory.  The model-card pages have no counterpart
 * for this entry point: it exists for callers such as plugins hosted by a
 * runtime that owns every device allocation, or code on a path where
 * cudaMalloc/cudaFree (which can synchronise the whole device) are not
 * allowed.  It takes the same arguments minus the workspace, and allocates
 * nothing: the split partials go to a file-scope device array of
 * PGD_STATIC_SCRATCH_BYTES inside the library.  The caller still owns q, the
 * pools, table, positions, sinks and out.
 *   - Returns PGD_ESCRATCH_LIMIT, with nothing launched, if these dims and
 *     options need more than PGD_STATIC_SCRATCH_BYTES of partials (that is,
 *     if pgd_paged_decode_workspace_bytes(dims, opts) exceeds it).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     outside any stream capture.
 *   - Every call on a device shares the one array, which keeps whatever the
 *     last call left there.  Nothing in it has to start at zero: every
 *     partial a call reads was written earlier in the same call.  Calls whose
 *     kernels can overlap on the GPU (different streams without ordering
 *     between them) race on the array and give wrong results; serialise them.
 * Results equal those of pgd_paged_decode_attention with the same options.
 */
PGD_API int pgd_paged_decode_attention_static(const pgd_dims* dims, const void* q,
                                              const void* k_pool, const void* v_pool,
                                              const int32_t* table, const int32_t* positions,
                                              const float* sinks, int32_t window, float scale,
                                              void* out, const pgd_decode_options* opts,
                                              pgd_stream_t stream);

/* Synchronises `stream`, then returns and clears the sticky device error word
 * of the current device (PGD_OK if none).  Returns PGD_ECUDA if the
 * synchronisation itself failed. */
PGD_API int pgd_get_device_error(pgd_stream_t stream);

/*
 * Self-test of failure detection, not part of the attention path: launches a
 * one-warp kernel whose two pipeline waits (an mbarrier phase and a shared
 * word, as the decode and prefill kernels use them) are never satisfied.
 * Each gives up after its limit (2 s), so the call takes about 4 s; the
 * kernel records PGD_EDEVICE_TIMEOUT and returns without faulting.  It then
 * runs what a decode split does after such a timeout on a fake row in shared
 * memory: as a row's only split it must zero the row's outputs, and as one of
 * two splits it must mark its partials so that the combine's merge gives
 * zero even though the other split is valid.
 *   outcome  device int32 [2]: [0] bit 0 / bit 1 set if the first / second
 *            wait was (wrongly) satisfied; [1] bit 0 set if the only-split
 *            case left a non-zero output, bit 1 if the merged two-split case
 *            did.  Both 0 after a correct run.
 * Read the status with pgd_get_device_error; the context stays usable.
 */
PGD_API int pgd_selftest_bounded_wait(int32_t* outcome, pgd_stream_t stream);

/* A static, human-readable name for a status code. */
PGD_API const char* pgd_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
PGD_API int pgd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PGD_H_ */
