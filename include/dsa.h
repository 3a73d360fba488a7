/*
 * dsa.h — C ABI of libdsa: query-aware dynamic block-sparse decode attention over a paged bf16
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * Sources restated (cited by title and section):
 *   [PSA]    "PSA: Progressive Sparse Attention — Algorithm and System Co-design for Efficient
 *             Attention in LLM Serving"
 *   [LServe] "LServe: Efficient Long-sequence LLM Serving with Unified Sparse Attention"
 *   [PRR]    "Predict, Reuse, and Repair: Accelerating Dynamic Sparse Attention for Long-Context
 *             LLM Decoding"
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller unless marked "host".  The
 *    library keeps no state between calls, allocates no memory, never synchronises the device and
 *    enqueues all work on `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 *  - Return value: DSA_OK (0) once the kernels are enqueued, or a negative DSA_ERR_* code when a
 *    host-side check fails, in which case nothing was enqueued; dsa_last_error() then returns a
 *    message for the calling thread.  Launch failures return DSA_ERR_CUDA.
 *  - Shapes: B = batch (requests), Hq = query heads, Hkv = KV heads, G = Hq / Hkv (query heads per
 *    KV head, 1..16), D = head_dim (128), p = page_size (multiple of 16, 16..256).
 *  - Softmax: logits s_t = scale * (q . k_t); m = max_t s_t (natural-log units); l = sum_t
 *    exp(s_t - m); O = sum_t exp(s_t - m) v_t / l.  An empty token set gives O = 0, m = -inf, l = 0.
 *  - Page ids read from the page table are checked against num_phys_pages; a bad id is skipped
 *    (its tokens contribute nothing) and DSA_STATUS_BAD_PAGE is OR-ed into *status when
 *    kv->status is non-NULL.
 *  - Scores use -inf for "no page here"; selection only ever picks pages with a score > -inf.
 *  - Alignment: the K/V pools, q and out (for the attention calls), metadata, partial records
 *    and workspaces must be 16-byte aligned; a misaligned pointer returns DSA_ERR_ALIGNMENT.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* dsa_stream_t; /* cudaStream_t */

enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = -1, /* null pointer, negative size, inconsistent shapes */
  DSA_ERR_ALIGNMENT = -2,   /* pointer not aligned as documented (16 B for bf16 pools) */
  DSA_ERR_UNSUPPORTED = -3, /* shape outside what the kernels implement (D != 128, G > 16, ...) */
  DSA_ERR_CUDA = -4,        /* a CUDA runtime / driver call failed */
  DSA_ERR_WORKSPACE = -5    /* workspace missing or smaller than the size query returned */
};

/* Bits a kernel may OR into kv->status (device int32).  Never set by a correct call. */
enum {
  DSA_STATUS_BAD_PAGE = 1, /* a page-table entry outside [0, num_phys_pages) was skipped */
  DSA_STATUS_OVERFLOW = 2, /* a list exceeded an internal capacity and was truncated */
  DSA_STATUS_TIMEOUT = 4   /* a bounded on-device wait gave up (the kernel returned early) */
};

enum { DSA_META_MINMAX = 0, DSA_META_MEAN = 1 };
enum { DSA_EMA_INIT = 0, DSA_EMA_UPDATE = 1 };
enum { DSA_PSA_NLEFT = 1 };

/*
 * The paged KV cache (the block/page KV cache of [PSA] §3.1 and [LServe] §3.2.1).
 *   k_pages, v_pages : bf16 [num_phys_pages][Hkv][p][D], 16-byte aligned, contiguous.  Token t of
 *                      request b is slot t % p of physical page page_table[b][t / p].
 *   page_table       : int32 [B][max_pages_per_seq].
 *   seq_lens         : int32 [B], tokens in the cache for each request (0 <= L_b <= p * max_pages).
 *   head_is_streaming: uint8 [Hkv] or NULL.  Non-zero marks a streaming (Lambda-mask) KV head
 *                      ([LServe] §4.1, dual cache §3.2.1): the dense-path calls (scoring,
 *                      selection, sparse attention, repair) skip those heads and leave their
 *                      outputs untouched; dsa_streaming_head_attn serves only those heads.
 *   status           : int32 [1] or NULL; device-detected problems are OR-ed into it.
 * The struct itself is read on the host during the call and not retained.
 */
typedef struct dsa_paged_kv {
  const void* k_pages;
  const void* v_pages;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const uint8_t* head_is_streaming;
  int32_t* status;
  int32_t batch;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;
  int32_t max_pages_per_seq;
  int32_t num_phys_pages;
} dsa_paged_kv;

/* Message for the last failed call on this host thread ("" if none). Host string, not owned. */
const char* dsa_last_error(void);
/* Library version string (host, static). */
const char* dsa_version(void);

/*
 * Per-page key metadata ([LServe] §4.2 and Figure 7: k_max / k_min kept with each page;
 * [PSA] §5: cuboid-mean block metadata).
 *   meta_kind    : DSA_META_MINMAX or DSA_META_MEAN.
 *   logical_page : tokens per logical page; divides p (g = p / logical_page sub-pages per page).
 *   meta (out)   : MINMAX -> bf16 [num_phys_pages][Hkv][g][D][2], pairs (max, min) per dimension;
 *                  MEAN   -> fp32 [num_phys_pages][Hkv][g][D].  16-byte aligned.
 * Every (request, page position j < ceil(L_b / p)) is processed: the physical page it maps to
 * gets the max/min (exact in bf16) or the fp32 mean of its valid tokens per logical sub-page.  A
 * sub-page with no valid token is written as zeros.  Physical pages no request reaches are left
 * untouched.  Streaming heads are processed too (the data is per page, not per head kind).
 */
int dsa_build_page_meta(const dsa_paged_kv* kv, int32_t meta_kind, int32_t logical_page,
                        void* meta, dsa_stream_t stream);

/*
 * Decode-time KV append ([LServe] §4.2: the page metadata is kept current as decoding adds
 * tokens): for every request b with L_b > 0, writes the token at position L_b - 1 -- kv->seq_lens
 * ALREADY counts it -- into its page of the pools (WRITTEN through kv->k_pages / kv->v_pages),
 * then recomputes the metadata of that page (every logical sub-page of it) exactly as
 * dsa_build_page_meta computes it, bit for bit.
 *   k_new, v_new : bf16 [B][Hkv][D], 16-byte aligned: the new token's key and value per KV head.
 *   meta         : as for dsa_build_page_meta, or NULL to write the KV only.  A caller keeping
 *                  several metadata buffers calls once per buffer (the KV write repeats
 *                  harmlessly).
 * The caller assigns page_table[b][(L_b - 1) / p] before a token that starts a new page.  A bad
 * page id skips the request and raises DSA_STATUS_BAD_PAGE.  One warp per (request, KV head).
 */
int dsa_append_kv(const dsa_paged_kv* kv, const void* k_new, const void* v_new,
                  int32_t meta_kind, int32_t logical_page, void* meta, dsa_stream_t stream);

/*
 * Page criticality ([LServe] §4.2: S^j = sum_i max(q_i kmax^j_i, q_i kmin^j_i); [PSA] §3.2:
 * CS = q . meta; [PRR] §5: one representative query per KV head for GQA).
 *   q            : bf16 [B][Hq][D].  The representative query of KV head h is the fp32 mean of
 *                  its G query heads h*G .. h*G+G-1.
 *   meta         : as written by dsa_build_page_meta with the same meta_kind / logical_page.
 *   scores (out) : fp32 [B][Hkv][score_stride]; score_stride >= max_pages_per_seq * g.  Logical
 *                  page j < ceil(L_b / logical_page) gets its score; slots beyond get -inf; the
 *                  whole row of a streaming head gets -inf.
 */
int dsa_score_pages(const dsa_paged_kv* kv, const void* q, const void* meta, int32_t meta_kind,
                    int32_t logical_page, float* scores, int32_t score_stride,
                    dsa_stream_t stream);

/*
 * Fixed-budget top-K page selection (the baseline selection of [PSA] §2.2 and [PRR] §2).
 *   scores      : fp32 [rows][stride]; entries 0..n-1 of each row are candidates; an entry
 *                 counts as valid when > -inf (NaN is invalid).
 *   k           : budget (>= 0).
 *   idx (out)   : int32 [rows][idx_stride], idx_stride >= k.  The min(k, #valid) highest-scoring
 *                 valid entries, ties to the lower index, written in ASCENDING index order;
 *                 slots past the count are set to -1.
 *   count (out) : int32 [rows].
 * n <= 32768.  One CTA per row.
 */
int dsa_select_topk(const float* scores, int32_t rows, int32_t n, int32_t stride, int32_t k,
                    int32_t* idx, int32_t idx_stride, int32_t* count, dsa_stream_t stream);

/*
 * Hierarchical paging selection ([LServe] §4.2): the score of physical page P is the max of the
 * logical scores P*g .. P*g+g-1 (restricted to < n_logical); then top-k_phys physical pages as in
 * dsa_select_topk (valid = > -inf, ties to the lower index, ascending output).  g = 1 is flat
 * top-K.  idx holds physical page POSITIONS within the request (units of p tokens).
 */
int dsa_select_hier(const float* logical_scores, int32_t rows, int32_t n_logical, int32_t stride,
                    int32_t g, int32_t k_phys, int32_t* idx, int32_t idx_stride, int32_t* count,
                    dsa_stream_t stream);

/*
 * PSA progressive threshold selection with fused attention ([PSA] §3.2, with the on-device
 * verification of §3.3: the stop decision never leaves the GPU).
 * For each dense (request b, KV head h): rank pages (block = one page of p tokens) by scores
 * (descending, ties to the lower index), visit them in rank order and stop after the first block
 * where, for every query head of the group, AS_acc / (AS_acc + AS_min) >= tau (AS = unnormalised
 * softmax mass of a block, AS_acc their running sum, AS_min the smallest seen), or after `cap`
 * blocks, or when the valid blocks run out.  With flags & DSA_PSA_NLEFT the rule reads
 * AS_acc / (AS_acc + N_left * AS_min), N_left = valid blocks not yet visited.
 *   scores       : fp32 [B][Hkv][score_stride] (one score per page, e.g. DSA_META_MEAN with
 *                  logical_page == p).
 *   tau          : 0 < tau <= 1.  cap >= 1.
 *   idx (out)    : int32 [B][Hkv][idx_stride], idx_stride >= cap: visited page positions in
 *                  visiting (rank) order; count (out) int32 [B][Hkv].
 *   out/m/l (out): fp32 [B][Hq][D], [B][Hq], [B][Hq]: attention over the visited blocks.
 * max_pages_per_seq <= 16384.
 */
int dsa_select_threshold(const dsa_paged_kv* kv, const void* q, const float* scores,
                         int32_t score_stride, float tau, int32_t cap, int32_t flags, float scale,
                         int32_t* idx, int32_t idx_stride, int32_t* count, float* out, float* m,
                         float* l, dsa_stream_t stream);

/*
 * Exact attention over the selected pages, split over pages (split-K) with a log-sum-exp merge
 * ([LServe] §3.3: iterate only the selected KV pages; [PRR] §3.3: the instrumented forward that
 * also writes m and l).
 *   idx, count   : int32 [B][Hkv][idx_stride], int32 [B][Hkv]: page positions (units of p) of
 *                  each dense row; order is free; positions >= ceil(L_b / p) or < 0 are skipped.
 *   out/m/l      : fp32 [B][Hq][D], [B][Hq], [B][Hq]; may be NULL when page_partials is given.
 *   page_partials: NULL, or fp32 [B][Hkv][idx_stride][G][D + 4]: for selected slot i the partial
 *                  record (O_0..O_{D-1}, m, l, 0, 0) of attention over that page alone (the
 *                  per-page partials PRR's exact repair merges).  Slots >= count are not written.
 *   num_splits   : 0 (default) = one persistent launch of one CTA per SM: the selected pages of
 *                  all dense rows are split into equal ranges, one per CTA; a row cut across
 *                  CTAs is merged by the CTA that finishes its last part (no second kernel);
 *                  > 0 = the pages of a row are spread over exactly this many CTAs and merged
 *                  by a second kernel.
 *   workspace    : device scratch of at least dsa_sparse_decode_attn_workspace_size() bytes,
 *                  16-byte aligned (may be NULL when that size is 0), ZERO-FILLED before its
 *                  first use: the persistent path keeps one ticket word per row in it, which
 *                  every completed call leaves at zero again (zero-fill it again after a call
 *                  that raised DSA_STATUS_TIMEOUT); the rest is scratch.
 */
int dsa_sparse_decode_attn(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                           int32_t idx_stride, const int32_t* count, float scale, float* out,
                           float* m, float* l, float* page_partials, int32_t num_splits,
                           void* workspace, size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_sparse_decode_attn_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride,
                                             int32_t num_splits);

/*
 * dsa_sparse_decode_attn without a caller-provided workspace (none of the three source pages has
 * a counterpart: this is a deployment convenience).  Some callers cannot call cudaMalloc: code
 * running inside a host framework that owns all device memory through its own allocator, and
 * latency-critical loops that cannot accept the device synchronisation cudaMalloc/cudaFree may
 * imply.  This variant always runs the explicit split-K path (per-split CTAs, then a merge
 * kernel): with the same num_splits > 0 it computes exactly what dsa_sparse_decode_attn computes;
 * with num_splits <= 0 it picks its own split count on that path (dsa_sparse_decode_attn's
 * default is its persistent kernel instead), so the two agree up to fp32 rounding.  It keeps the
 * split-K partial records in a fixed 4 MiB device array inside the library, which every GPU that
 * loads the library holds until exit.
 *   - Allocates nothing; calls no cudaMalloc/cudaFree or allocating library routine.
 *   - The first call on each device looks up the array's device address (cudaGetSymbolAddress,
 *     with that device current) and caches it; make that first call before any stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU (e.g. on two streams)
 *     race and corrupt each other's results; serialise them.  The array needs no clearing: every
 *     record a call reads is written earlier in the same call.
 *   - When rows * splits * G * 528 bytes exceeds the array (dsa_sparse_decode_attn_noalloc_
 *     max_bytes()), the call returns DSA_ERR_UNSUPPORTED and enqueues nothing.
 *   - out/m/l are required (no page_partials mode).
 */
int dsa_sparse_decode_attn_noalloc(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                                   int32_t idx_stride, const int32_t* count, float scale,
                                   float* out, float* m, float* l, int32_t num_splits,
                                   dsa_stream_t stream);
size_t dsa_sparse_decode_attn_noalloc_max_bytes(void);

/*
 * PRR repair and merge ([PRR] §3.3 repair kernel and recurrence).  Given the speculative set P
 * (spec_idx/spec_count, ASCENDING and unique) whose per-page partials a previous
 * dsa_sparse_decode_attn wrote to page_partials (same idx_stride = spec_stride), and the true set
 * A (true_idx/true_count, ASCENDING and unique): attention is computed only for the missed pages
 * M = A \ P, and merged with the partials of
 *     superset == 0: P ∩ A          -> out = attention over A exactly,
 *     superset != 0: all of P       -> out = attention over P ∪ A.
 *   out/m/l (out): fp32 [B][Hq][D], [B][Hq], [B][Hq].
 *   workspace    : at least dsa_repair_merge_workspace_size() bytes.
 */
int dsa_repair_merge(const dsa_paged_kv* kv, const void* q, const int32_t* spec_idx,
                     int32_t spec_stride, const int32_t* spec_count, const float* page_partials,
                     const int32_t* true_idx, int32_t true_stride, const int32_t* true_count,
                     int32_t superset, float scale, float* out, float* m, float* l,
                     void* workspace, size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_repair_merge_workspace_size(const dsa_paged_kv* kv, int32_t true_stride);

/*
 * Streaming heads ([LServe] §4.1, Lambda-shaped mask): for every KV head marked in
 * kv->head_is_streaming, exact attention of its G query heads over tokens
 * [0, min(sink, L_b)) ∪ [max(0, L_b - local), L_b).  Writes out/m/l rows of those heads only.
 */
int dsa_streaming_head_attn(const dsa_paged_kv* kv, const void* q, int32_t sink_tokens,
                            int32_t local_tokens, float scale, float* out, float* m, float* l,
                            dsa_stream_t stream);

/*
 * Dense and streaming heads in one launch ([LServe] §3.2-§4.1: one sparse-attention pass serves
 * both head kinds): the dense KV heads attend their selected pages exactly as the persistent path
 * of dsa_sparse_decode_attn does, and the KV heads marked in kv->head_is_streaming attend tokens
 * [0, min(sink_tokens, L_b)) ∪ [max(0, L_b - local_tokens), L_b) as dsa_streaming_head_attn does
 * -- the streaming rows' pages join the same stream-K cut of work over one CTA per SM.
 * With kv->head_is_streaming NULL it equals dsa_sparse_decode_attn (persistent path).
 *   idx/count/idx_stride : the dense rows' selections (streaming rows' entries are not read).
 *   out/m/l (out)        : every query head, 16-byte aligned out.
 *   workspace            : dsa_sparse_decode_attn_workspace_size(kv, idx_stride, 0) bytes,
 *                          zero-filled before its first use (as for dsa_sparse_decode_attn).
 */
int dsa_hybrid_decode_attn(const dsa_paged_kv* kv, const void* q, const int32_t* idx,
                           int32_t idx_stride, const int32_t* count, int32_t sink_tokens,
                           int32_t local_tokens, float scale, float* out, float* m, float* l,
                           void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * KV8 pages (an own 8-bit page format; [LServe] §3.2.1 and its quantised KV pages motivate it:
 * fewer bytes per selected page).  Every K and V row (one token of one KV head) of the pool is
 * stored as 128 e4m3 values with one fp32 scale: scale = max_i |x_i| / 448 (448 = the largest
 * finite e4m3 value) and byte_i = e4m3(x_i / scale), rounded to nearest even, saturating; a row of
 * zeros gets scale 0 and zero bytes.  A value decodes as e4m3_value(byte) * scale.
 * Layout: one contiguous block of 264 p bytes per (physical page P, KV head h), at offset
 * (P * Hkv + h) * 264 p: the K codes [p][128], the V codes [p][128], the K scales fp32 [p], the V
 * scales fp32 [p] -- so the attention brings a selected page with one bulk copy.  In the code row
 * of token slot r the 16 codes of dims 16 c .. 16 c + 15 are stored at bytes 16 (c ^ (r mod 8))
 * .. +15 (a bank-spreading permutation for the attention's operand loads).
 *   kv8 (out) : dsa_kv8_bytes(kv) bytes, 16-byte aligned.
 * Every physical page is converted (the bf16 pools are read, not changed).
 */
int dsa_quantize_kv8(const dsa_paged_kv* kv, void* kv8, dsa_stream_t stream);
size_t dsa_kv8_bytes(const dsa_paged_kv* kv);

/*
 * Sparse decode attention over KV8 pages: as the persistent path of dsa_sparse_decode_attn (exact
 * attention of every dense head's query group over the tokens of its selected pages, one stream-K
 * launch) over the KV8 blocks: the tensor-core products take the e4m3 codes as f16 (exact) with
 * the query in f16 (|q| below 65504), each logit times its token's K scale and each probability
 * times its token's V scale (rounded to f16 for the P.V product).  kv->k_pages / v_pages are not
 * read (may be NULL); the page table, lengths and shapes are.  Streaming heads are skipped.
 *   workspace : dsa_sparse_decode_attn_kv8_workspace_size(kv, idx_stride) bytes, zero-filled
 *               before its first use (as for dsa_sparse_decode_attn).
 */
int dsa_sparse_decode_attn_kv8(const dsa_paged_kv* kv, const void* kv8, const void* q,
                               const int32_t* idx, int32_t idx_stride, const int32_t* count,
                               float scale, float* out, float* m, float* l, void* workspace,
                               size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_sparse_decode_attn_kv8_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride);

/*
 * KV4 pages (an own 4-bit page format; [LServe] §2.2 decodes over 4-bit KV, the W4A8KV4 setting
 * it builds on, without giving a format).  Every K and V row of the pool is stored as 128 integer
 * codes with one fp32 scale: scale = max_i |x_i| / 7 and code_i = round(x_i / scale) (fp32
 * division, ties to even) in [-7, 7], kept as the nibble code_i + 8, dims 2i and 2i + 1 in the low
 * and high half of byte i; a row of zeros gets scale 0 and codes 0.  A value decodes as
 * (nibble - 8) * scale.
 * Layout: one contiguous block of 136 p bytes per (physical page P, KV head h), at offset
 * (P * Hkv + h) * 136 p: the K codes [p][64], the V codes [p][64], the K scales fp32 [p], the V
 * scales fp32 [p].  The 64-byte code row of token slot r is stored at row r ^ ((r >> 1) & 1) (in
 * every other pair of rows the two swap places: a bank-spreading permutation for the attention's
 * operand loads).
 *   kv4 (out) : dsa_kv4_bytes(kv) bytes, 16-byte aligned.
 * Every physical page is converted (the bf16 pools are read, not changed).
 */
int dsa_quantize_kv4(const dsa_paged_kv* kv, void* kv4, dsa_stream_t stream);
size_t dsa_kv4_bytes(const dsa_paged_kv* kv);

/*
 * Sparse decode attention over KV4 pages: as dsa_sparse_decode_attn_kv8 over KV4 blocks (the codes
 * enter the tensor-core products as f16, exact; logits times the token's K scale, probabilities
 * times its V scale, rounded to f16 for the P.V product).
 *   workspace : dsa_sparse_decode_attn_kv4_workspace_size(kv, idx_stride) bytes, zero-filled
 *               before its first use (as for dsa_sparse_decode_attn).
 */
int dsa_sparse_decode_attn_kv4(const dsa_paged_kv* kv, const void* kv4, const void* q,
                               const int32_t* idx, int32_t idx_stride, const int32_t* count,
                               float scale, float* out, float* m, float* l, void* workspace,
                               size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_sparse_decode_attn_kv4_workspace_size(const dsa_paged_kv* kv, int32_t idx_stride);

/*
 * PRR EMA predictor ([PRR] §3.1) fused with the speculative-set selection ([PRR] §3.4 with a fixed
 * budget |P| = k_pred).
 *   IS           : fp32 [rows][stride], the true scores of this step (entries 0..n-1; -inf =
 *                  no page).
 *   ell, v       : fp32 [rows][stride] level and trend, updated in place:
 *                  DSA_EMA_INIT  : ell = IS, v = 0;
 *                  DSA_EMA_UPDATE: v = beta (IS - ell) + (1 - beta) v, ell = alpha IS + (1 - alpha)
 *                                  ell (both read the previous ell).
 *                  Entries with IS = -inf get ell = -inf, v = 0.
 *   pred (out)   : fp32 [rows][stride] or NULL: the next step's prediction ell + gamma v (-inf
 *                  where ell = -inf).
 *   pred_idx/pred_count (out): top-k_pred of the prediction, as dsa_select_topk (may be NULL
 *                  when k_pred == 0).
 */
int dsa_ema_predict_update(const float* IS, int32_t rows, int32_t n, int32_t stride, float* ell,
                           float* v, int32_t mode, float alpha, float beta, float gamma,
                           float* pred, int32_t k_pred, int32_t* pred_idx,
                           int32_t pred_idx_stride, int32_t* pred_count, dsa_stream_t stream);

/*
 * Calibration of the EMA predictor ([PRR] §3.2): every (alpha, beta, gamma) of the 80-point grid
 * runs the predictor of dsa_ema_predict_update over a trajectory of true score vectors, and is
 * rated by the mean score-weighted hit rate
 *     H = mean over t = 1..steps-1 of  sum_{j in A_t ∩ P_t} IS_t[j] / sum_{j in A_t} IS_t[j]
 * (1 for a step whose A_t scores sum to 0), where A_t = top-k of IS_t and P_t = top-k_pred of the
 * prediction made from steps 0..t-1 (step 0 initialises the state); both selections rank as
 * dsa_select_topk does.  The grid point with the largest H wins, ties to the lower point.
 * Grid point c (0..79): alpha = 0.2 (1 + c / 20), beta = 0.1 (1 + (c / 4) % 5),
 * gamma = 0.25 (c % 4) -- alpha outermost, gamma innermost.  One CTA per (row, grid point);
 * the parameters are fp32.
 *   traj      : fp32 [steps][rows][stride], IS_t of row r at traj[(t * rows + r) * stride];
 *               entries 0..n-1 are pages (-inf = no page).  1 <= n <= min(stride, 16384).
 *   H (out)   : fp32 [rows][80].
 *   best (out): int32 [rows], the winning grid point.
 *   1 <= k, k_pred <= 256; steps >= 1 (steps = 1 rates every point 0 and picks point 0).
 *   workspace : dsa_calibrate_ema_workspace_size(steps, rows, n, k) bytes, 16-byte aligned, its
 *               first 4 * rows bytes ZERO-FILLED before the first use (each completed call
 *               leaves them zero-filled); the rest is scratch: A_t of every (step, row), selected
 *               once because it does not depend on the grid point, and the predictor state of
 *               every (row, grid point), 640 * n bytes per row.
 * Two launches: the top-k selection of A_t over the whole trajectory, then the grid.
 */
#define DSA_CALIB_POINTS 80
int dsa_calibrate_ema(const float* traj, int32_t steps, int32_t rows, int32_t n, int32_t stride,
                      int32_t k, int32_t k_pred, float* H, int32_t* best, void* workspace,
                      size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_calibrate_ema_workspace_size(int32_t steps, int32_t rows, int32_t n, int32_t k);

/*
 * One whole PRR decode step t >= 1 in a single launch ([PRR] §3 end to end: speculation over the
 * predicted set P_t (§3.4), the true selection A_t, the predictor update (§3.1), repair of the
 * missed pages and the merge (§3.3)).  It computes exactly what this sequence computes:
 *   dsa_score_pages(q, meta, DSA_META_MINMAX, logical_page = page_size)     -> scores (= IS_t)
 *   dsa_select_topk(scores, n = stride, k)                                  -> idx/count (= A_t)
 *   dsa_sparse_decode_attn(P_t = spec_idx/spec_count, page_partials)        -> page_partials
 *   dsa_ema_predict_update(scores, DSA_EMA_UPDATE, k_pred)                  -> ell, trend, pred,
 *                                                                              next_idx/next_count
 *   dsa_repair_merge(P_t, page_partials, A_t, superset)                     -> out/m/l
 * with scores, A_t, the EMA state and P_{t+1} bit for bit and out/m/l up to fp32 rounding.  One
 * launch of one CTA per SM, all resident at once (the step assumes no other stream holds SMs for
 * long while it runs; its waits are bounded and raise DSA_STATUS_TIMEOUT), launched as a
 * programmatic dependent of the previous kernel in the stream: its CTAs are scheduled while that
 * kernel finishes and wait for it before reading global memory.  No CTA waits for the whole grid:
 * the worker CTAs (all CTAs but the task CTAs when the grid holds at least four CTAs per task,
 * else every CTA) score equal shares of the (request, KV head, page) slots, every CTA attends its
 * pages of P_t, and the selections, the repair and the merges wait only for their own row's
 * counters.
 *   args->q            : bf16 [B][Hq][D], 16-byte aligned.  Device memory, or page-locked host
 *                        memory mapped for the device (cudaHostAlloc / cudaHostRegister): the
 *                        kernel then reads the query over the host link itself, no copy needed.
 *   args->meta         : DSA_META_MINMAX metadata built with logical_page == page_size.
 *   args->scores (out) : fp32 [B][Hkv][stride]; max_pages_per_seq <= stride <= 32768.
 *   args->ell, trend   : fp32 [B][Hkv][stride], EMA level and trend, updated in place.
 *   args->pred (out)   : fp32 [B][Hkv][stride] or NULL.
 *   args->spec_idx/spec_count : P_t, int32 [B][Hkv][k_pred] ASCENDING and unique, int32 [B][Hkv].
 *   args->page_partials (out) : fp32 [B][Hkv][k_pred][G][D + 4], 16-byte aligned: the per-page
 *                        records of P_t (a slot whose page lies outside the request holds the
 *                        empty part).
 *   args->idx/count (out)     : A_t, int32 [B][Hkv][k] ascending, int32 [B][Hkv].
 *   args->next_idx/next_count (out): P_{t+1}, int32 [B][Hkv][k_pred], int32 [B][Hkv]; must not
 *                        alias spec_idx/spec_count (double-buffer them across steps).
 *   args->out/m/l (out): fp32 [B][Hq][D], [B][Hq], [B][Hq].  Like q, they may be mapped
 *                        page-locked host memory, which the kernel writes directly.
 *   1 <= k, k_pred <= 256.  kv->head_is_streaming must be NULL.
 *   workspace          : dsa_prr_step_workspace_size(kv) bytes, 16-byte aligned.  Its first
 *                        dsa_prr_step_counter_bytes(kv) bytes hold per-row counters and must be
 *                        ZERO-FILLED before the first use; every call that completes leaves them
 *                        at zero again.  If a call raised DSA_STATUS_TIMEOUT they must be
 *                        zero-filled again.  Next come per-row candidate hints that each call
 *                        reads and rewrites for the next one (any contents are safe: they only
 *                        decide how fast A_t is found; zero them with the counters to start
 *                        clean), then scratch the call writes before it reads.
 * A_t is selected exactly, but its search is speculative: while scoring, the kernel lists the pages
 * of each row that score at or above the row's hint (the key ranked k + k/2 at the previous call);
 * when at least k pages are listed, the row's k best are among them and only the list is ranked.
 * Otherwise (the first call, scores that fell below the hint, a worker CTA listing more than 15 pages
 * of a row, or more than 512 listed pages) every entry of the row is ranked.  P_{t+1} is searched the same way from a bound, the k_pred-th
 * largest prediction over P_t's pages, falling back to ranking every entry when it does not hold.
 */
typedef struct dsa_prr_step_args {
  const void* q;
  const void* meta;
  float* scores;
  int32_t stride;
  float* ell;
  float* trend;
  float alpha;
  float beta;
  float gamma;
  float* pred;
  const int32_t* spec_idx;
  const int32_t* spec_count;
  int32_t k_pred;
  float* page_partials;
  int32_t* idx;
  int32_t* count;
  int32_t k;
  int32_t* next_idx;
  int32_t* next_count;
  int32_t superset;
  float scale;
  float* out;
  float* m;
  float* l;
} dsa_prr_step_args;
int dsa_prr_step(const dsa_paged_kv* kv, const dsa_prr_step_args* args, void* workspace,
                 size_t workspace_bytes, dsa_stream_t stream);
size_t dsa_prr_step_workspace_size(const dsa_paged_kv* kv);
size_t dsa_prr_step_counter_bytes(const dsa_paged_kv* kv);

/*
 * Log-sum-exp merge of partial records ([PRR] §3.3 recurrence, applied to all parts at once).
 *   partials : fp32 [rows][num_parts][G][D + 4] records (O, m, l, 0, 0); a record with l == 0 is
 *              the identity.
 *   out/m/l  : fp32 [rows * G][D], [rows * G], [rows * G].
 */
int dsa_merge_partials(const float* partials, int32_t rows, int32_t num_parts, int32_t group,
                       int32_t head_dim, float* out, float* m, float* l, dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
