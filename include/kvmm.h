/*
 * kvmm.h -- C ABI of libkvmm: query-aware MinMax page selection and sparse
 * paged GQA decode attention on NVIDIA GB300 (sm_103a).
 *
 * The method follows two pages:
 *   FlexiCache: Leveraging Temporal Stability of Attention Heads for
 *   Efficient KV Cache Management (MLSys'26; blog summary), sections
 *   "Core method, 2. MinMax-metadata page scoring",
 *   "Core method, 3. Periodic reranking and incremental promotion",
 *   "Core method, 1. Stability-differentiated placement" (attention over the
 *   top-K pages only) and "System design, head-level block table";
 *   KVDrive: A Holistic Multi-Tier KV Cache Management System for
 *   Long-Context LLM Inference, "Background and key observations" (Quest
 *   scores a page by multiplying the query with the keys' channel-wise
 *   minimum and maximum).
 *
 * Terms.  A unit is one (batch b, layer l, KV head h).  Each unit owns a
 * sequence of logical pages of T tokens; page p holds tokens
 * [p*T, (p+1)*T).  A head-level block table maps (b, l, h, p) to a physical
 * page of the shared K and V pools; the entry KVMM_NULL_BLOCK (-1) marks a
 * page that is not resident and is never dereferenced.  The G = Hq / Hkv
 * query heads h*G .. h*G+G-1 share KV head h.
 *
 * Conventions for every call:
 *   - All array pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing; scratch comes from a caller workspace.
 *   - Arrays are dense, row-major, in the layouts given below; bf16 values
 *     are raw 16-bit patterns (kvmm_bf16).  bf16 arrays and workspaces must
 *     be 16-byte aligned, int32 and float arrays 4-byte aligned; a
 *     violation returns KVMM_INVALID_ARG.
 *   - Work is enqueued on the caller's stream and runs asynchronously.  The
 *     return value only reports host-side argument checks and launch
 *     errors: KVMM_OK means the work was enqueued.
 *   - Faults found on the device never trap: they OR a KVMM_ERR_* bit into
 *     the caller's device word *err (which the caller zeroes and reads after
 *     synchronising) and the offending page or row is skipped.
 *   - NaN or Inf inputs are not supported; they give undefined values but
 *     no fault.
 *   - Calls that share a workspace, or write the same outputs, must not
 *     run concurrently (calls on one stream never do).
 */
#ifndef KVMM_H
#define KVMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvmm_bf16;              /* raw bf16 bit pattern */
typedef struct CUstream_st* kvmm_stream; /* a cudaStream_t; NULL = legacy default stream */

typedef enum kvmm_status {
    KVMM_OK = 0,
    KVMM_INVALID_ARG = 1,        /* null/misaligned pointer, index out of range, bad flag */
    KVMM_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported set (see kvmm_shape) */
    KVMM_WORKSPACE_TOO_SMALL = 3,
    KVMM_CUDA_ERROR = 4          /* a CUDA runtime call or kernel launch failed */
} kvmm_status;

/* Bits OR-ed into the caller's device error word. */
#define KVMM_ERR_NULL_BLOCK 1   /* a page that had to be read maps to the null block */
#define KVMM_ERR_OUT_OF_RANGE 2 /* a table entry >= n_phys, a selected page >= the unit's page
                                   count, a sequence longer than Pmax*T, or more rows than given */
#define KVMM_ERR_TIMEOUT 4      /* a bounded wait on an in-flight copy gave up (never expected) */

#define KVMM_NULL_BLOCK (-1)

/* Shape shared by all calls.
 *   B      batch size                      L     layers held in the arrays
 *   Hq     query heads per layer           Hkv   KV heads per layer (Hq % Hkv == 0, G <= 8)
 *   D      head dimension (64 or 128)      T     tokens per page (16 or 32)
 *   Pmax   logical pages per unit held by the block table and the metadata
 *          (1 <= Pmax <= 32768)
 *   Kmax   capacity of a unit's selection list (1 <= Kmax <= 32768)
 *   n_phys physical pages in each of the K and V pools                    */
typedef struct kvmm_shape {
    int32_t B, L, Hq, Hkv, D, T, Pmax, Kmax;
    int64_t n_phys;
} kvmm_shape;

/* Array layouts (all row-major):
 *   k_pool           [n_phys][T][D]            bf16, a page's keys token by token
 *   v_pool           [n_phys][D][T]            bf16, a page's values dimension by dimension
 *                                              (the value cache layout of paged serving engines)
 *   block_table      [B][L][Hkv][Pmax]         int32, -1 = null block
 *   meta             [B][L][Hkv][Pmax][2][D]   bf16, [..][0][d] = min, [..][1][d] = max
 *   q                [B][Hq][D]                bf16 (the layer being decoded)
 *   seq_len          [B]                       int32, tokens in the sequence (<= Pmax*T)
 *   rescore_mask     [L][Hkv]                  uint8, nonzero = rescore this step
 *   sel_idx          [B][L][Hkv][Kmax]         int32 logical pages, ascending
 *   sel_cnt          [B][L][Hkv]               int32
 *   out              [B][Hq][D]                float
 *   lse              [B][Hq]                   float (natural log)                 */

/* ------------------------------------------------------------------------
 * kv_minmax_update -- append token rows to their pages and refresh the
 * per-page, per-channel key MinMax metadata of every page they touch.
 *
 * FlexiCache, "Core method, 2. MinMax-metadata page scoring": each KV page
 * keeps the per-channel minimum and maximum of its keys; the metadata lives
 * apart from the K/V pages (so it stays on the GPU even when the page does
 * not) and is indexed by logical page.
 *
 * For each batch b, with n = tok_end[b] - tok_begin[b] (0 <= n <= n_new):
 *   - if new_k and new_v are given ([B][Hkv][n_new][D] bf16 each, token by
 *     token), token tok_begin[b] + j of every KV head of `layer` takes row j
 *     of new_k / new_v, written into its physical page through block_table
 *     (keys as a row of the page, values as a column of the page's [D][T]);
 *   - if both are NULL nothing is written (metadata rebuild only; n_new is
 *     then only an upper bound on n and may be as large as Pmax*T);
 *   - for every logical page p with [p*T, (p+1)*T) meeting
 *     [tok_begin[b], tok_end[b]), meta[b][layer][h][p] is recomputed over the
 *     page's tokens below tok_end[b] (tok_end[b] is the sequence length after
 *     the update).  min/max compare by value with -0 below +0.
 * Null or out-of-range table entries set their error bit and are skipped;
 * n > n_new sets KVMM_ERR_OUT_OF_RANGE and clamps n.
 */
kvmm_status kv_minmax_update(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* new_k,
                             const kvmm_bf16* new_v, int32_t n_new, const int32_t* tok_begin,
                             const int32_t* tok_end, kvmm_bf16* k_pool, kvmm_bf16* v_pool,
                             const int32_t* block_table, kvmm_bf16* meta, int32_t* err,
                             kvmm_stream stream);

/* ------------------------------------------------------------------------
 * page_score_topk -- score every page of every rescored unit of `layer`
 * against the query and keep the K best pages.
 *
 * FlexiCache, "Core method, 2. MinMax-metadata page scoring" (estimate from
 * the page's key bounds the largest dot product the query can reach and keep
 * the top-K pages per (layer, KV head)); KVDrive, "Background and key
 * observations" (Quest: query times channel-wise key min and max).
 *
 * For a unit with P = ceil(seq_len[b] / T) pages and query heads g of its
 * group, page p scores
 *     s_g(p) = sum_d max(q_g[d] * min_p[d], q_g[d] * max_p[d])
 * (the largest q_g.k over the box [min_p, max_p]); the unit's score is
 * sum_g s_g(p) when group_reduce = 0 (the default) or max_g s_g(p) when
 * group_reduce = 1.  Scores are computed in fp32.  The min(K, P) highest
 * scoring pages are written to sel_idx[b][layer][h][0..) in ascending page
 * order, ties going to the lower page index, and sel_cnt to their count.
 *
 * rescore_mask (may be NULL = every unit) selects the units scored this
 * step; the others keep sel_idx / sel_cnt untouched (FlexiCache, "Core
 * method, 3": stable heads reuse their previous top-K between reranks).
 * scores_out, if not NULL, is [B][Hkv][Pmax] float and receives the fp32
 * scores of rescored units (pages >= P are not written).
 * workspace must hold kvmm_workspace_size(shape, 0) bytes of device memory;
 * it needs no initialisation (the call writes every score it reads) and
 * holds nothing between calls.
 * Requires 1 <= K <= Kmax; a sequence longer than Pmax*T sets
 * KVMM_ERR_OUT_OF_RANGE and is scored over its first Pmax pages.
 * The work is one launch: a cluster of CTAs streams a pair of units'
 * metadata, scores it and selects on chip (the workspace is not touched);
 * shapes whose per-unit buffers do not fit one CTA (beyond about 9,500
 * pages) run a scoring kernel and a selection kernel through the workspace.
 * flags: 0, or KVMM_EARLY_READS: the caller guarantees that no kernel still
 * running when this launch starts writes seq_len, the layer's rescore_mask
 * row or its metadata rows (after a kvmm call, the guarantee is about that
 * call alone; see decode_layer).  The launch then starts streaming the
 * metadata while that kernel drains, and waits for it before it reads q or
 * writes anything but error bits.  The two-kernel fallback always waits.
 */
kvmm_status page_score_topk(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                            const kvmm_bf16* meta, const int32_t* seq_len,
                            const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                            int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                            void* workspace, size_t workspace_bytes, uint32_t flags, int32_t* err,
                            kvmm_stream stream);

/* ------------------------------------------------------------------------
 * page_score_topk_static_scratch -- page_score_topk without a caller
 * workspace.  The pages have no counterpart to this call; it exists for
 * callers that cannot allocate device memory when they need the selection:
 * an engine whose pool allocator has already claimed all of HBM, a runtime
 * with no device-allocation hook of its own, or a decode loop that must not
 * pay cudaMalloc's implicit device synchronisation.  Those callers still own
 * and pass every input and output; only the scratch moves into the library.
 *
 * Same arguments, semantics and results as page_score_topk, minus
 * workspace / workspace_bytes.  The scratch is one fixed 4 MiB array in the
 * library's own device memory (every GPU that loads libkvmm holds it until
 * the process exits): it takes B * Hkv * Pmax <= 1,048,576 scores; a larger
 * shape returns KVMM_WORKSPACE_TOO_SMALL and nothing runs.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress,
 * once per device, cached); make that first call before any stream
 * capture.  The cached address belongs to the device's current context: a
 * process that calls cudaDeviceReset on a device must not call this entry
 * point on that device again.  Every call on a device shares the one array
 * and leaves its last contents in it (nothing needs to start at zero: each
 * call writes every score it reads), so calls whose kernels overlap on the
 * GPU (different streams, or concurrent host threads) race and give wrong
 * selections; serialise them (calls on one stream never overlap).
 */
kvmm_status page_score_topk_static_scratch(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                           const kvmm_bf16* meta, const int32_t* seq_len,
                                           const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                                           int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                                           int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * sparse_paged_decode_attn -- GQA decode attention of every query head of
 * `layer` over the valid tokens of its KV head's selected pages only.
 *
 * FlexiCache, "Core method, 1. Stability-differentiated placement" (decode
 * attention runs over the top-K pages even where the full KV is resident)
 * and "System design, head-level block table" (pages are found through
 * [batch, layer, head, logical_block]; null entries are never read).
 *
 * For query head g of KV head h in batch b, over the tokens t < seq_len[b]
 * of the pages sel_idx[b][layer][h][0 .. sel_cnt):
 *     z_t = sm_scale * (q_g . k_t)
 *     out[b][g]  = sum_t exp(z_t - m) v_t / sum_t exp(z_t - m),  m = max_t z_t
 *     lse[b][g]  = m + log(sum_t exp(z_t - m))
 * accumulated in fp32.  sm_scale <= 0 means 1/sqrt(D).  A unit with no
 * valid token yields out = 0 and lse = -inf.  Each unit's selection is
 * split over the CTAs of one thread-block cluster, which merge their
 * partial results by log-sum-exp in distributed shared memory.  With
 * num_splits = 0 the launch shape is automatic: two units share a cluster
 * as large as the GPU holds in one wave (kvmm_auto_splits gives its CTAs
 * per unit), and a unit's pages stream into the slots the previous unit's
 * pages free.  An explicit num_splits runs one unit a cluster of that many
 * CTAs (clamped to [1, min(16, Kmax)]; a value the device cannot co-schedule
 * returns KVMM_UNSUPPORTED_SHAPE).  A selected page whose entry is null or
 * out of range, or whose index is >= the unit's page count, sets its error
 * bit and contributes nothing.  lse may be NULL.  workspace /
 * workspace_bytes are not used by this call (kept for the stable signature)
 * and may be NULL / 0.
 * flags: 0, or KVMM_EARLY_READS (automatic launch shape only): the caller
 * guarantees that no kernel still running when this launch starts writes
 * seq_len or the layer's block-table rows.  The launch then computes its
 * units' extents and copies their table rows while that kernel drains, and
 * waits for it before it reads q, the selections or the pools.  A
 * page_score_topk just before writes only selections and scores, so a
 * decode loop may set the flag whenever the table changes between steps.
 */
kvmm_status sparse_paged_decode_attn(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                     const kvmm_bf16* k_pool, const kvmm_bf16* v_pool,
                                     const int32_t* block_table, const int32_t* seq_len,
                                     const int32_t* sel_idx, const int32_t* sel_cnt,
                                     float sm_scale, int32_t num_splits, float* out, float* lse,
                                     void* workspace, size_t workspace_bytes, uint32_t flags,
                                     int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * topk_promotion_diff -- after a rerank, list the pages that entered and
 * left each rescored unit's top-K.
 *
 * FlexiCache, "Core method, 3. Periodic reranking and incremental
 * promotion": only (current top-K minus previous top-K) is transferred; and
 * "System design, head-level block table" (physical blocks of evicted pages
 * are reused for promoted pages), which the evicted list serves.
 *
 * For every unit of `layer` with rescore_mask set (NULL = all):
 *     promoted = cur \ prev,   evicted = prev \ cur
 * both ascending, from the ascending lists prev_idx[0..prev_cnt) and
 * cur_idx[0..cur_cnt) (layouts of sel_idx / sel_cnt).  Units not rescored
 * get promoted_cnt = evicted_cnt = 0.  evicted / evicted_cnt may be NULL.
 * total_promoted, if not NULL, is a single device int32 to which the call
 * atomically adds the number of promoted pages.  With commit != 0, prev is
 * then overwritten by cur for the rescored units, so prev always holds the
 * last committed selection.  Lists that are not strictly ascending, or
 * counts outside [0, Kmax], set KVMM_ERR_OUT_OF_RANGE and the unit's output
 * counts are 0.
 */
kvmm_status topk_promotion_diff(const kvmm_shape* shape, int32_t layer,
                                const uint8_t* rescore_mask, int32_t* prev_idx,
                                int32_t* prev_cnt, const int32_t* cur_idx,
                                const int32_t* cur_cnt, int32_t commit, int32_t* promoted,
                                int32_t* promoted_cnt, int32_t* evicted, int32_t* evicted_cnt,
                                int32_t* total_promoted, int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * page_score_topk_attn -- page_score_topk followed by
 * sparse_paged_decode_attn on the new selection.
 *
 * FlexiCache, "Core method, 2. MinMax-metadata page scoring" (score every
 * page from its key bounds, keep the top-K per layer and KV head) and
 * "Core method, 1" / "System design, head-level block table" (attend over
 * the selected pages only, through the head-level table).  One launch of
 * the clustered kernel decode_layer runs, with nothing appended: a cluster
 * streams its units' metadata, scores and selects on chip, then streams the
 * selected pages.  Shapes whose per-unit buffers do not fit that kernel
 * (long page tables) run two kernels instead: the scoring kernel, then an
 * attention kernel whose CTAs select their unit's pages from the scores
 * themselves before streaming them.
 *
 * Arguments, layouts and results are those of the two calls: sel_idx /
 * sel_cnt / scores_out of rescored units as page_score_topk writes them (the
 * others keep their selection, which the attention then uses), and out /
 * lse as sparse_paged_decode_attn writes them with its automatic split
 * count.  workspace as for page_score_topk (the one-launch kernel does not
 * touch it).  When the selection does not fit the attention CTA's shared
 * memory either (Pmax beyond about 30,000 pages), the call runs
 * page_score_topk and then sparse_paged_decode_attn (same results).
 */
kvmm_status page_score_topk_attn(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                 const kvmm_bf16* meta, const kvmm_bf16* k_pool, const kvmm_bf16* v_pool,
                                 const int32_t* block_table, const int32_t* seq_len,
                                 const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                                 float sm_scale, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out,
                                 float* out, float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * decode_layer -- one layer of a decode step in one launch: append the new
 * tokens and refresh their pages' MinMax (kv_minmax_update), score every
 * page and select the top K (page_score_topk), attend over the selected
 * pages (sparse_paged_decode_attn).
 *
 * FlexiCache, "Core method, 2. MinMax-metadata page scoring" (the bounds are
 * kept up to date as pages fill; every page is scored; the top-K pages of
 * each layer and KV head are kept) and "Core method, 1" / "System design,
 * head-level block table" (attention over the selected pages only).
 *
 * Arguments and results are those of the three calls: new_k / new_v
 * ([B][Hkv][n_new][D], or both NULL to append nothing), n_new, tok_begin,
 * tok_end as for kv_minmax_update (the appended rows are written to the
 * pools and their pages' MinMax refreshed before those pages are scored);
 * rescore_mask, K, group_reduce, sel_idx, sel_cnt, scores_out as for
 * page_score_topk; sm_scale, out, lse as for sparse_paged_decode_attn.
 * seq_len already counts the appended tokens.  Two units (batch, KV head)
 * share one thread-block cluster, which scores, selects and attends entirely
 * on chip: no workspace.  For shapes whose buffers do not fit one CTA's shared
 * memory (long page tables), the call runs kv_minmax_update and then
 * page_score_topk_attn instead, which need workspace (as for page_score_topk;
 * otherwise workspace may be NULL and is not used).
 *
 * flags: 0, or KVMM_DECODE_EARLY_READS.  By default the launch reads nothing
 * before the kernel launched just before it on the stream has finished
 * (programmatic dependent launch lets it be scheduled meanwhile).  With
 * KVMM_DECODE_EARLY_READS the caller guarantees that no kernel still running
 * when this launch starts writes anything this call reads of seq_len,
 * tok_begin, tok_end, rescore_mask (the layer's row), block_table and meta
 * (the layer's rows).  The launch then reads those while that kernel drains
 * (the units' extents, their table rows, the first metadata rows) and waits
 * for it before it reads q, new_k, new_v, the pools or the kept selections,
 * and before it writes anything but the error bits of out-of-range lengths
 * or token ranges (atomic ORs into err).
 * Every kvmm kernel lets the next launch start only after its own wait for
 * its predecessor has returned, so when the kernel just before this call is
 * a kvmm call (or a kernel launched without programmatic dependent launch),
 * it is the only kernel that can still be running: the guarantee is then
 * about that one kernel.  A decode loop meets it when those arrays change
 * only between steps or by the call itself and consecutive decode_layer
 * calls on the stream are for different layers (the layers of a step back
 * to back, two or more layers), or when the query projection runs just
 * before.  Two decode_layer calls for the SAME layer back to back (a
 * one-layer loop) do not meet it: the first writes the metadata row of the
 * page it appends to, which the second would read early; leave the flag off
 * there.  Other bits return KVMM_INVALID_ARG.  The two-kernel fallback always
 * waits.
 */
#define KVMM_EARLY_READS 1u
#define KVMM_DECODE_EARLY_READS KVMM_EARLY_READS
kvmm_status decode_layer(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q, const kvmm_bf16* new_k,
                         const kvmm_bf16* new_v, int32_t n_new, const int32_t* tok_begin, const int32_t* tok_end,
                         kvmm_bf16* k_pool, kvmm_bf16* v_pool, const int32_t* block_table, kvmm_bf16* meta,
                         const int32_t* seq_len, const uint8_t* rescore_mask, int32_t K, int32_t group_reduce,
                         float sm_scale, int32_t* sel_idx, int32_t* sel_cnt, float* scores_out, float* out,
                         float* lse, void* workspace, size_t workspace_bytes, uint32_t flags, int32_t* err,
                         kvmm_stream stream);

/* ------------------------------------------------------------------------
 * The mean-key scorer: KVDrive's page representative, beside MinMax.
 *
 * KVDrive, "Method details": the KV cache is split into blocks and each
 * page's mean key is its representative in the index (higher-level
 * centroids then group similar pages).  The score of page p for query head
 * g is q_g . mean_p, on D channels where MinMax reads 2D.
 *
 * kv_meankey_update -- mean [B][L][Hkv][Pmax][D] bf16: for every logical
 * page meeting [tok_begin[b], tok_end[b]) (tok_begin NULL = from 0), the
 * mean of the page's keys below tok_end[b]: their fp32 sum in token order,
 * divided by their count, rounded to bf16 (nearest even).  Null or
 * out-of-range table entries set their error bit and the page is skipped;
 * a range outside [0, Pmax*T] sets KVMM_ERR_OUT_OF_RANGE and is clamped.
 */
kvmm_status kv_meankey_update(const kvmm_shape* shape, int32_t layer, const int32_t* tok_begin,
                              const int32_t* tok_end, const kvmm_bf16* k_pool, const int32_t* block_table,
                              kvmm_bf16* mean, int32_t* err, kvmm_stream stream);

/* page_score_topk_mean -- page_score_topk with the mean key as the page's
 * row: s_g(p) = q_g . mean_p (fp32), group sum (or max), top K with the same
 * ties, order, rescore mask, scores_out and workspace as page_score_topk.
 */
kvmm_status page_score_topk_mean(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                 const kvmm_bf16* mean, const int32_t* seq_len, const uint8_t* rescore_mask,
                                 int32_t K, int32_t group_reduce, int32_t* sel_idx, int32_t* sel_cnt,
                                 float* scores_out, void* workspace, size_t workspace_bytes, int32_t* err,
                                 kvmm_stream stream);

/* ------------------------------------------------------------------------
 * The centroid level of KVDrive's index over the pages' mean keys.
 *
 * KVDrive, "Method details": each page's mean key is its representative and
 * higher-level centroids group similar pages; "the trade-off between block
 * size and centroid count": the centroid count is kept proportional to the
 * context (a fixed number of pages per centroid), and the grouping by
 * similarity matches a spatial blocking's accuracy with half the centroids.
 * The page names no clustering algorithm.  The one built here, per unit:
 * Lloyd's k-means over the unit's P pages' mean keys, started from spatial
 * blocks (page p in centroid p / R, n_c = ceil(P / R) centroids):
 *   - assignment: a page joins the centroid of least squared Euclidean
 *     distance, accumulated as fmaf(x, x, acc) in fp32 over the channels in
 *     order (x = mean - centroid), ties to the lower centroid;
 *   - update: a centroid becomes the bf16 (nearest even) of the fp32 mean of
 *     its pages' mean keys, summed in page order; one with no page keeps its
 *     value.
 *
 * kv_centroid_build -- the spatial blocks, then n_iter Lloyd iterations
 * (0 <= n_iter <= 64; 0 leaves the spatial blocking), for every unit of
 * `layer`.  mean [B][L][Hkv][Pmax][D] as kv_meankey_update writes it.
 * Outputs, with Cmax = ceil(Pmax / R):
 *   cent       [B][L][Hkv][Cmax][D] bf16   the centroids (rows >= n_c untouched)
 *   assign     [B][L][Hkv][Pmax]    int32  each page's centroid (pages >= P untouched)
 *   member_off [B][L][Hkv][Cmax + 1] int32 centroid j's pages are
 *   members    [B][L][Hkv][Pmax]    int32  members[member_off[j] .. member_off[j + 1]), ascending
 * Requires 1 <= R <= Pmax; shapes whose per-unit buffers do not fit a CTA
 * (about Pmax + Cmax > 56,000) return KVMM_UNSUPPORTED_SHAPE.
 */
kvmm_status kv_centroid_build(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* mean, const int32_t* seq_len,
                              int32_t R, int32_t n_iter, kvmm_bf16* cent, int32_t* assign, int32_t* member_off,
                              int32_t* members, int32_t* err, kvmm_stream stream);

/* page_score_topk_centroid -- the two-level selection over the index: score
 * the unit's n_c centroids like pages (q_g . c, the group summed or, with
 * group_reduce = 1, maxed; fp32), expand the M best (ties to the lower
 * centroid; all when M >= n_c), score the pages of those centroids by their
 * mean keys the same way, and keep the K best of those pages (ties to the
 * lower page) in sel_idx, ascending, with their count in sel_cnt.
 * rescore_mask as for page_score_topk (units not rescored keep their
 * selection).  R is the build's.  centroid_scores_out [B][Hkv][Cmax] and
 * scores_out [B][Hkv][Pmax] (written for the expanded pages only) may be
 * NULL.  Requires 1 <= M, 1 <= K <= Kmax; shapes whose selection buffers do
 * not fit a CTA (Pmax beyond about 16,000) return KVMM_UNSUPPORTED_SHAPE.
 */
kvmm_status page_score_topk_centroid(const kvmm_shape* shape, int32_t layer, const kvmm_bf16* q,
                                     const kvmm_bf16* mean, const int32_t* seq_len, int32_t R, const kvmm_bf16* cent,
                                     const int32_t* member_off, const int32_t* members, const uint8_t* rescore_mask,
                                     int32_t M, int32_t K, int32_t group_reduce, int32_t* sel_idx, int32_t* sel_cnt,
                                     float* centroid_scores_out, float* scores_out, int32_t* err,
                                     kvmm_stream stream);

/* ------------------------------------------------------------------------
 * block_table_update -- apply the changed entries of the head-level block
 * table: block_table[idx[i]] = val[i], i = 0 .. n-1.
 *
 * FlexiCache, "System design, head-level block table": with dirty tracking
 * only the changed regions of the [batch, layer, head, logical_block] table
 * are synchronised, not the whole four-dimensional table every step.  Here
 * the changed entries themselves are the delta: idx (int64 flat indices into
 * [B][L][Hkv][Pmax]) and val (a physical block, or -1 for the null block)
 * may live in device memory or in host memory the device can read (a pinned
 * staging buffer filled by the host scheduler), so only those 12 bytes per
 * entry cross the host link.  Indices must be distinct (a dirty set); with
 * repeats the entry takes one of the values.  An index outside the table or
 * a value outside [-1, n_phys) sets KVMM_ERR_OUT_OF_RANGE and that update is
 * skipped.  n = 0 launches nothing.
 */
kvmm_status block_table_update(const kvmm_shape* shape, const int64_t* idx, const int32_t* val, int32_t n,
                               int32_t* block_table, int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * promote_pages -- after a rerank, bring each rescored unit's promoted pages
 * from the host KV store into the GPU pools, in the physical blocks its
 * evicted pages free, and rewrite the block table.
 *
 * FlexiCache, "Core method, 3. Periodic reranking and incremental
 * promotion" (only the promoted pages are transferred), "Core method, 4.
 * Overlapping transfer and compute" (a UVA kernel reads the pinned host KV
 * directly, with a bounded grid, so that it leaves the SMs to decoding) and
 * "System design, head-level block table" (physical block reuse: evicted
 * pages' blocks go to promoted pages; evicted entries keep their place and
 * point at the null block).
 *
 * For every unit of `layer` with rescore_mask set (NULL = all), promoted
 * [0..np) and evicted [0..ne) ascending (as topk_promotion_diff writes
 * them, same layouts as sel_idx / sel_cnt), m = min(np, ne):
 *   - i < m: phys = block_table[evicted[i]]; block_table[evicted[i]] = -1;
 *     block_table[promoted[i]] = phys; logical page promoted[i] of the host
 *     store is copied into pool page phys;
 *   - i >= m of evicted: block_table[evicted[i]] = -1, and its block is
 *     returned in freed[i - m] (when given; -1 if the entry was skipped),
 *     freed_cnt = ne - m;
 *   - i >= m of promoted: no block is free; the entry is left as it was.
 * moved [B][L][Hkv] (may be NULL) receives m minus the skipped pairs.
 * host_k / host_v: [B][L][Hkv][Pmax][T][D] / [B][L][Hkv][Pmax][D][T] bf16
 * (each logical page laid out as a pool page), in host memory the device
 * can address: pinned, or pageable where the device reads pageable host
 * memory (a coherent host link).  freed [B][L][Hkv][Kmax] and freed_cnt
 * [B][L][Hkv] may be NULL.  max_ctas bounds the grid (0: 16).
 * An evicted entry that is null or outside the pool sets
 * KVMM_ERR_NULL_BLOCK / KVMM_ERR_OUT_OF_RANGE and its pair moves nothing;
 * pages outside [0, Pmax) or counts outside [0, Kmax] set
 * KVMM_ERR_OUT_OF_RANGE.  Decode of the same units must not run
 * concurrently (stream order suffices).
 */
kvmm_status promote_pages(const kvmm_shape* shape, int32_t layer, const uint8_t* rescore_mask,
                          const int32_t* promoted, const int32_t* promoted_cnt, const int32_t* evicted,
                          const int32_t* evicted_cnt, const kvmm_bf16* host_k, const kvmm_bf16* host_v,
                          kvmm_bf16* k_pool, kvmm_bf16* v_pool, int32_t* block_table, int32_t* moved,
                          int32_t* freed, int32_t* freed_cnt, int32_t max_ctas, int32_t* err, kvmm_stream stream);

/* ------------------------------------------------------------------------
 * Temporal stability of each (layer, KV head): offline profiling that
 * classifies heads as stable or unstable.
 *
 * FlexiCache, "Core insight: attention heads differ in temporal stability":
 * the top-K page set of each head is recorded at every decode step; sets a
 * few steps apart are compared with the Random-Corrected Overlap (RCO),
 * which is 1 for identical sets and 0 for the overlap random sets would
 * have; RCO is aggregated over a window of W steps into a per-head
 * stability score, and the least stable 25% of the heads are classed
 * unstable (they are rescored every step, see rescore_mask).
 *
 * The pages print no formula.  The reading used here: for sets A, B drawn
 * from P pages,
 *     RCO(A, B) = (|A n B| - |A||B|/P) / (min(|A|, |B|) - |A||B|/P)
 * where |A||B|/P is the expected overlap of random subsets of those sizes
 * and min(|A|, |B|) the largest possible one; RCO = 1 when the two are
 * equal (every page selected, or P = 0).  When the sequence grew between
 * the two steps, P is the later (larger) page count.
 * ------------------------------------------------------------------------
 *
 * topk_history_record -- store layer `layer`'s current selections (every
 * layer's when layer = -1, in one launch) in slot `slot` (0 <= slot < W) of
 * a history ring of W steps:
 *     hist_idx   [W][B][L][Hkv][Kmax] int32   <- sel_idx  (ascending pages)
 *     hist_cnt   [W][B][L][Hkv]       int32   <- sel_cnt
 *     hist_pages [W][B]               int32   <- ceil(seq_len[b] / T), the
 *                page count the selections were taken over (seq_len clamped
 *                to [0, Pmax*T], out-of-range values set KVMM_ERR_OUT_OF_RANGE
 *                when err is given).
 * A decode step records every layer into the same slot (step mod W).
 */
kvmm_status topk_history_record(const kvmm_shape* shape, int32_t layer, const int32_t* sel_idx,
                                const int32_t* sel_cnt, const int32_t* seq_len, int32_t W, int32_t slot,
                                int32_t* hist_idx, int32_t* hist_cnt, int32_t* hist_pages, int32_t* err,
                                kvmm_stream stream);

/* topk_stability_rco -- stability of every unit and head from the last n
 * recorded steps of the ring (the newest in slot `head`, the one before in
 * slot head - 1 mod W, ...), comparing selections `lag` steps apart.
 *     rco_unit  [B][L][Hkv] float: the mean of RCO(S_t, S_{t+lag}) over the
 *               n - lag pairs t = 0 .. n - lag - 1 (t steps before the newest);
 *     stability [L][Hkv] float (may be NULL): the mean of rco_unit over b;
 *     unstable  [L][Hkv] uint8 (may be NULL): 1 for the round(unstable_frac *
 *               L * Hkv) heads of lowest stability (ties: lower l * Hkv + h
 *               first), else 0.
 * Requires 1 <= n <= W, 0 <= head < W, 1 <= lag < n, 0 <= unstable_frac <= 1
 * (else KVMM_INVALID_ARG), n <= 1024 and L * Hkv <= 4096 (else
 * KVMM_UNSUPPORTED_SHAPE).
 * A recorded count outside [0, Kmax], or a page count outside [0, Pmax], sets
 * KVMM_ERR_OUT_OF_RANGE and is clamped; a recorded page outside [0, Pmax)
 * sets it and is not counted.  Selections must be ascending and distinct (as
 * sel_idx is); their overlap is counted exactly.  Sums run in double.
 */
kvmm_status topk_stability_rco(const kvmm_shape* shape, const int32_t* hist_idx, const int32_t* hist_cnt,
                               const int32_t* hist_pages, int32_t W, int32_t n, int32_t head, int32_t lag,
                               float unstable_frac, float* rco_unit, float* stability, uint8_t* unstable,
                               int32_t* err, kvmm_stream stream);

/* Workspace bytes that page_score_topk and page_score_topk_attn need
 * (sparse_paged_decode_attn needs none; num_splits is accepted for the
 * stable signature and ignored).  Returns 0 for an unsupported shape. */
size_t kvmm_workspace_size(const kvmm_shape* shape, int32_t num_splits);

/* Number of splits per unit that sparse_paged_decode_attn uses for
 * num_splits = 0 on the current device (0 for an unsupported shape). */
int32_t kvmm_auto_splits(const kvmm_shape* shape);

/* The launch shape of decode_layer's one-launch kernel for this shape on the
 * current device.  kvmm_decode_layer_units: (batch, KV head) units a cluster
 * of CTAs takes, 2 when their buffers fit shared memory, else 1 (long
 * sequences: the scores of a unit take 4 bytes a page).
 * kvmm_decode_layer_cluster: CTAs per cluster, the most whose clusters are
 * all resident at once.  Both are 0 when decode_layer does not launch that
 * kernel for the shape (an unsupported shape, or buffers that do not fit
 * even for one unit; it then runs kv_minmax_update and page_score_topk_attn). */
int32_t kvmm_decode_layer_cluster(const kvmm_shape* shape);
int32_t kvmm_decode_layer_units(const kvmm_shape* shape);

/* Static text for a status code. */
const char* kvmm_status_string(kvmm_status status);

/* Text of the CUDA error behind the calling thread's last KVMM_CUDA_ERROR
 * ("no CUDA error" if there was none). */
const char* kvmm_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVMM_H */
