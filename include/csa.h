/*
 * libcsa: the decode step of a C4 hybrid-sparse-attention layer on GB300 (sm_103a).
 *
 * The operation (web pages, cited by title and section):
 *   [V4-deploy] "DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "V4 到底改了啥":
 *       every layer attends a sliding window of the last 128 raw tokens (SWA) plus
 *       either C4 (4:1 compression of the KV, top-512 sparse selection) or C128
 *       (128:1 compression, attended densely).
 *     sec. "Kernel 層一堆狠活": SWA and the extra (C4/C128) attention in ONE call;
 *       Flash Compressor (load -> score -> softmax -> weighted sum -> store in one
 *       on-chip pass); Lightning TopK (top-512 of 256K candidates at 1M context by
 *       a cluster-of-8 radix select instead of a global sort).
 *   [Day-0] "SGLang 如何为 DeepSeek V4 打造「Day-0」推理加速",
 *     sec. "创新 2：Flash Compressor + Lightning TopK": per-CTA 10-bit histograms,
 *       reduced inside the cluster to a threshold, then a local scatter of the
 *       entries above it; warp-local softmax for C4, one CTA per group for C128.
 *     sec. "创新 1：ShadowRadix": one virtual token-slot space projected onto the
 *       physical pools ("shadow" pages) -- adopted here as the paging convention.
 *   The pages print no formulas; the problem statement fixes them:
 *     gate      s_i = kv_i . w_gate + b_pos[i]               (i = position in the group)
 *     score[g]  = sum_h w_h * ReLU(q_idx[h] . k_idx[g])       (fp32, fixed order below)
 *     top-k     by descending score, ties to the lower index.
 *
 * Shapes fixed in this version: latent D = 512 (K = V = the latent row, bf16),
 * index dim 128, ratio in {4, 128}, k <= 2048, swa <= 128, query heads
 * 1 <= H <= 128 (padded to the 128-row tensor-core tile inside), index heads
 * 1 <= Hi <= 16.
 *
 * Conventions for every entry point
 *  - Pointers are DEVICE pointers unless stated otherwise; the caller owns all
 *    memory (inputs, outputs, workspace).  libcsa never allocates, frees or
 *    synchronises on these calls: work is enqueued on `stream` and the call
 *    returns.  The stream is a cudaStream_t passed as void* (0 = legacy default).
 *  - Argument/shape errors return synchronously, before anything is enqueued.
 *    A failed launch returns CSA_ERR_CUDA.  Errors a kernel detects (a page id
 *    outside the pool, a bounded wait that ran out) are OR-ed into a sticky
 *    per-device status word read with csa_read_device_status(); kernels never
 *    trap or assert.
 *  - Alignment: every bf16/fp8 row buffer and query pointer must be 16-byte
 *    aligned, fp32/int32 arrays 4-byte aligned; page strides are multiples of 16.
 */
#ifndef CSA_H_
#define CSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned pointer */
    CSA_ERR_UNSUPPORTED = 2,   /* outside the fixed limits above */
    CSA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
    CSA_ERR_TIMEOUT = 4,       /* device status: a bounded wait ran out */
    CSA_ERR_DEVICE_BOUNDS = 5, /* device status: a page id / index outside its pool (access skipped) */
    CSA_ERR_WORKSPACE = 6      /* workspace missing or smaller than the *_workspace_size query */
} csa_status;

typedef enum { CSA_BF16 = 0, CSA_FP8_E4M3 = 1, CSA_FP32 = 2 } csa_dtype;

/*
 * A paged row buffer (the ShadowRadix "physical pool" view).
 * Logical row r lives in logical page p = r / rows_per_page, slot s = r % rows_per_page;
 * its bytes start at base + P * page_stride_bytes + s * row_bytes, where
 * P = page_table[p] (device int32) or P = p when page_table is NULL (contiguous).
 * row_bytes is fixed by the tensor (1024 for a bf16 latent row, 256 for a bf16
 * index key, 128 for an fp8 index key).  n_pages bounds P (device-checked).
 */
typedef struct {
    void* base;
    const int32_t* page_table; /* device, or NULL */
    int32_t rows_per_page;     /* >= 1 */
    int64_t page_stride_bytes; /* >= rows_per_page * row_bytes, multiple of 16 */
    int64_t n_pages;           /* physical pages in the pool */
} csa_paged;

/*
 * Stage 1, standalone (prefill): softmax-gated ratio:1 compression
 * ([V4-deploy] "Kernel 層一堆狠活", Flash Compressor; [Day-0] "创新 2").
 * For each group j in [first_group, first_group + n_groups): tokens
 * ratio*j .. ratio*j+ratio-1 of kv_raw (bf16 [n_tokens, 512]),
 *   s_i = kv_i . w_gate + b_pos[i], a = softmax(s), c_j = sum_i a_i kv_i,
 * fp32 arithmetic, written as bf16 (RN) to row j of kv_c_out.
 * w_gate: fp32 [512]; b_pos: fp32 [ratio].  ratio 4: one warp per group;
 * ratio 128: one CTA per group.  Requires (first_group + n_groups) * ratio <= n_tokens.
 */
csa_status csa_compress(csa_paged kv_raw, int64_t n_tokens, int32_t ratio, const float* w_gate,
                        const float* b_pos, int64_t first_group, int64_t n_groups, csa_paged kv_c_out,
                        void* stream);

/*
 * Stage 2: index score of every candidate ([V4-deploy] "Kernel 層一堆狠活", indexer).
 * q_idx bf16 [Hi, 128] (contiguous), w_h fp32 [Hi], k_idx rows ([G, 128], bf16 or
 * fp8-e4m3 per k_dtype; paged tables need rows_per_page % 16 == 0), scores fp32 [G].
 * Bit-exact fixed order:
 *   Q[j] = q[32j]*k[32j], then Q[j] = fma(q[32j+i], k[32j+i], Q[j]) for i = 1..31  (j = 0..3)
 *   dot = (Q[0] + Q[2]) + (Q[1] + Q[3])
 *   acc = 0; acc = fma(w_h, dot > 0 ? dot : +0, acc) for h = 0..Hi-1
 */
csa_status csa_index_score(const void* q_idx, const float* w_h, int32_t Hi, csa_paged k_idx, csa_dtype k_dtype,
                           int64_t G, float* scores, void* stream);

/*
 * Stage 2 as brackets, on the tensor cores ([V4-deploy] "Kernel 層一堆狠活": the indexer's
 * q.k products are a dense contraction): for every candidate g, lower[g] <= s[g] <= upper[g],
 * s the fixed-order score of csa_index_score.  The dots q_h . k_g come from tcgen05 MMAs (bf16
 * operands, fp32 accumulation); the half-width is
 *   e_g = 2^-13 * max_j |k_gj| * sum_h |w_h| * ||q_h||_1 + 1e-30   (rounded up),
 * which covers the fixed-order chains' rounding (at most 33 * 2^-24 of sum_j |q_hj k_gj|) and
 * an MMA accumulation error of up to 2^-14 of the same sum.  A non-finite input or a bound past
 * 1e30 gives (-inf, +inf); a row whose page id is out of range gives [0, 0] and the device
 * status CSA_ERR_DEVICE_BOUNDS.  Arguments as csa_index_score; k_dtype must be CSA_BF16
 * (otherwise CSA_ERR_UNSUPPORTED); lower is nullable, both fp32 [G], 4-byte aligned.
 * csa_decode takes this form in speculative verify with bf16 index keys (2 <= n_q <= 4, Hi <= 16):
 * one pass over the keys serves every query position, and the select rescores in the fixed
 * order only the candidates whose upper bound reaches the histogram bin (top 12 or 13 bits of
 * the key) of the k-th largest lower bound, so its top k is the fixed-order score's top k.
 */
csa_status csa_index_score_bounds(const void* q_idx, const float* w_h, int32_t Hi, csa_paged k_idx,
                                  csa_dtype k_dtype, int64_t G, float* lower, float* upper, void* stream);

/*
 * Stage 3: top-k ([Day-0] "创新 2", Lightning TopK: per-CTA histograms reduced to
 * a threshold, then a scatter of the entries above it).
 * scores fp32 [G] -> idx_out int32 [k]: the indices of the min(k, G) largest
 * scores ordered by (score desc, index asc), then -1 padding.  Scores compare
 * through the order-preserving key (-0 == +0; key = bits ^ (sign ? ~0 : 1<<31)).
 * keys_out (nullable) uint32 [k] receives those keys (0 for padding).
 * Radix select over the key's digits.  Up to 4,194,304 scores per request: CTAs of 2,048
 * scores each count the first digit and add their counts into a histogram in global
 * memory (L2 atomics); a wide grid then compacts every slice's winners and threshold
 * candidates, and a finish kernel in which every CTA ranks its own slice's entries writes
 * the output (no CTA gathers them all).  Above that size the call takes the single-cluster
 * form of csa_topk_cluster.
 * workspace: device, 16-byte aligned, at least csa_topk_workspace_size(1, G, k) bytes,
 * owned by the caller, its contents overwritten (no state is kept between calls).
 * 1 <= k <= 2048, G <= 2^31 - 1.  CSA_ERR_WORKSPACE when it is missing or small.
 */
size_t csa_topk_workspace_size(int32_t B, int64_t max_G, int32_t k);
csa_status csa_topk(const float* scores, int64_t G, int32_t k, int32_t* idx_out, uint32_t* keys_out,
                    void* workspace, size_t ws_bytes, void* stream);

/*
 * Batched stage 3 over a ragged batch: request b owns scores[offsets[b] .. offsets[b+1])
 * (offsets: device int64 [B+1]), writes idx_out[b*k .. b*k+k) (indices local to
 * the request).  max_G: host-side bound on every request's length.  workspace:
 * csa_topk_workspace_size(B, max_G, k) bytes.
 */
csa_status csa_topk_batched(const float* scores, const int64_t* offsets, int32_t B, int64_t max_G, int32_t k,
                            int32_t* idx_out, uint32_t* keys_out, void* workspace, size_t ws_bytes,
                            void* stream);

/*
 * Stage 3, single-cluster form: the output of csa_topk_batched (indices sorted by (score
 * desc, index asc), keys_out optional, -1 padding), computed by one thread-block cluster
 * per request as the pages describe Lightning TopK ([Day-0] "创新 2": per-CTA histograms
 * reduced inside the cluster to the threshold, then the entries above it scattered).  Each
 * CTA of the cluster (up to 16, a power of two, about 16,384 scores each) owns a contiguous
 * slice and keeps its winners and threshold candidates in its own shared memory; every
 * radix digit is counted in each CTA's shared memory and the cluster's counts are summed
 * through distributed shared memory; CTA 0 ranks the union.  csa_topk and
 * csa_topk_batched take this form by themselves above 4,194,304 scores per request; this
 * entry point takes it at any size.  offsets: device int64 [B+1], or NULL with B = 1 for
 * one request of max_G scores.  No workspace; nothing is allocated.
 */
csa_status csa_topk_cluster(const float* scores, const int64_t* offsets, int32_t B, int64_t max_G, int32_t k,
                            int32_t* idx_out, uint32_t* keys_out, void* stream);

/*
 * Stage 4: one attention over the selected compressed entries plus the last
 * W = min(swa, n_tokens) raw tokens under a single softmax ([V4-deploy]
 * "Kernel 層一堆狠活": FlashMLA's one call for SWA + extra attention).
 * q bf16 [H, 512]; kv_c: compressed pool (bf16 rows); sel int32 [n_sel] row ids
 * into kv_c (entries < 0 are padding and ignored), or NULL for all rows
 * 0..n_sel-1 (dense C128); kv_raw: raw pool (bf16 rows, n_tokens of them).
 * For head h: l_j = scale * q_h . K_j, o_h = softmax(l) . V (K = V = the row);
 * out bf16 [H, 512]; lse fp32 [H] (natural log, nullable).
 * tcgen05 tensor cores (M = 128 padded heads, 64-key tiles), keys split across
 * CTAs and merged by log-sum-exp.  Workspace: csa_sparse_attn_workspace_size().
 */
csa_status csa_sparse_attn(const void* q, int32_t H, float scale, csa_paged kv_c, const int32_t* sel, int32_t n_sel,
                           csa_paged kv_raw, int64_t n_tokens, int32_t swa, void* out, float* lse, void* workspace,
                           size_t ws_bytes, void* stream);
size_t csa_sparse_attn_workspace_size(int32_t H, int32_t n_sel, int32_t swa);

/*
 * Context-parallel split of one request ([Day-0] "3.1 长上下文预填充：Context Parallelism
 * (CP)": the tokens are shared out over ranks and the indexer's results meet in one
 * exchange).  Rank r holds the contiguous candidate range [lo_r, hi_r) of the request (its
 * index keys and compressed rows), the last rank also the raw rows of the SWA window.  A
 * decode step:
 *   1. each rank: csa_index_score over its range, csa_topk of those scores with keys_out
 *      (sorted; indices local to the range);
 *   2. exchange: all-gather the R lists of k (key, index) pairs, in rank order;
 *   3. each rank: csa_topk_merge -> the exact global top k (every rank gets the same set),
 *      and the rows of it that the rank holds;
 *   4. each rank: csa_sparse_attn_partial over those rows (the last rank adding the window);
 *   5. exchange: gather the R partials; csa_attn_merge -> the step's output.
 * The result equals the single-device step: the same selected set (bit-exact), the same
 * attention within rounding.
 */

/*
 * The exact top k of the union of R sorted local top-k lists.  keys uint32 [R * k] (from
 * csa_topk's keys_out: order-preserving keys), idx int32 [R * k] (csa_topk's indices, local to
 * each rank's range; < 0: padding), both rank-major.  rank_lo: device int64 [R + 1], rank r
 * holding the global candidates [rank_lo[r], rank_lo[r+1]) (increasing ranges).  Output,
 * each nullable: idx_out int32 [k] global indices by (score desc, index asc), -1 padding;
 * keys_out uint32 [k]; sel_local int32 [k]: g - rank_lo[rank] for the selected g that rank
 * `rank` holds, -1 for the others (the selection argument of csa_sparse_attn_partial on that
 * rank).  workspace: csa_topk_merge_workspace_size(R, k) bytes.  R * k <= 4,194,304,
 * k <= 2048.  An index outside its rank's range sets CSA_ERR_DEVICE_BOUNDS and is dropped.
 */
size_t csa_topk_merge_workspace_size(int32_t R, int32_t k);
csa_status csa_topk_merge(const uint32_t* keys, const int32_t* idx, const int64_t* rank_lo, int32_t R, int32_t k,
                          int32_t rank, int32_t* sel_local, int32_t* idx_out, uint32_t* keys_out, void* workspace,
                          size_t ws_bytes, void* stream);

/*
 * Stage 4 over one rank's share of the keys, as a mergeable partial: the arguments of
 * csa_sparse_attn, but the output is o_part fp32 [H, 512] (the normalised rows,
 * softmax(l) . V over this share) and lse_part fp32 [H] (natural log of the share's sum of
 * exp(l)).  An empty share (n_sel = 0 or only -1 entries, and no window) gives zero rows
 * and lse = -inf.  Workspace: csa_sparse_attn_workspace_size(H, n_sel, swa).
 */
csa_status csa_sparse_attn_partial(const void* q, int32_t H, float scale, csa_paged kv_c, const int32_t* sel,
                                   int32_t n_sel, csa_paged kv_raw, int64_t n_tokens, int32_t swa, float* o_part,
                                   float* lse_part, void* workspace, size_t ws_bytes, void* stream);

/*
 * Log-sum-exp merge of R partials over disjoint key sets of the same heads: o_parts fp32
 * [R, H, 512], lse_parts fp32 [R, H] -> out bf16 [H, 512] = sum_r e^(lse_r - M) O_r / L and
 * lse fp32 [H] (nullable) = M + ln L, with M = max_r lse_r, L = sum_r e^(lse_r - M).
 * Partials with lse = -inf contribute nothing; if all are empty, out = 0 and lse = -inf.
 */
csa_status csa_attn_merge(const float* o_parts, const float* lse_parts, int32_t R, int32_t H, void* out, float* lse,
                          void* stream);

/*
 * The fused decode step over a ragged batch of B requests ([V4-deploy] "V4 到底改了啥",
 * "Kernel 層一堆狠活"; [Day-0] "创新 2").  Per request b, with N = n_tokens[b],
 * G = N / ratio, done = n_groups_done[b]:
 *   1. compress groups [done, G) of the raw KV into the compressed pool (stage 1);
 *   2. ratio 4:   score all G candidates (stage 2), select the top k (stage 3),
 *                 attend the selection + SWA (stage 4);
 *      ratio 128: attend all G compressed entries + SWA (stage 4, dense).
 * Paging: one page table per request (row b of page_table, page_table_stride
 * int32 entries apart) maps logical page p (raw tokens p*rpp .. p*rpp+rpp-1,
 * rpp = raw_rows_per_page) to a physical page id.  With c_page_table == NULL the
 * compressed pool and the index-key pool are SHADOW pools: they use the same
 * physical page id and hold rpp / ratio rows per page (needs rpp % ratio == 0).
 * Otherwise c_page_table (row b, c_page_table_stride apart) pages them with
 * c_rows_per_page rows per page.
 * Per-request lengths live in device memory (so the call can be captured in a
 * CUDA graph once and replayed); max_tokens is a host-side bound used to size grids.
 */
typedef struct {
    int32_t B, ratio, H, Hi, k, swa;
    float scale;
    csa_dtype k_dtype;           /* index-key storage: CSA_BF16 or CSA_FP8_E4M3 */
    int64_t max_tokens;          /* >= every n_tokens[b] */
    const int64_t* n_tokens;     /* device [B], multiples of ratio, >= ratio */
    const int64_t* n_groups_done;/* device [B], 0 <= done <= G */
    /* pools shared by the batch */
    void* kv_raw;                /* bf16 rows of 1024 B */
    int32_t raw_rows_per_page;
    int64_t raw_page_stride;     /* bytes */
    void* kv_c;                  /* compressed pool, bf16 rows of 1024 B (written for pending groups) */
    int64_t c_page_stride;       /* bytes */
    const void* k_idx;           /* index keys (ratio 4), rows of 256 B (bf16) or 128 B (fp8) */
    int64_t kidx_page_stride;    /* bytes */
    int64_t n_pages;             /* physical pages in every pool (bounds check) */
    const int32_t* page_table;   /* device [B, page_table_stride] */
    int64_t page_table_stride;
    const int32_t* c_page_table; /* device [B, c_page_table_stride] or NULL (shadow paging) */
    int64_t c_page_table_stride;
    int32_t c_rows_per_page;     /* used when c_page_table != NULL */
    int64_t c_n_pages;           /* used when c_page_table != NULL */
    /* layer weights */
    const float* w_gate;         /* fp32 [512] */
    const float* b_pos;          /* fp32 [ratio] */
    /* per-request queries (B * n_q entries with speculative verify, see n_q) */
    const void* q;               /* bf16 [B, H, 512] */
    const void* q_idx;           /* bf16 [B, Hi, 128] (ratio 4) */
    const float* w_h;            /* fp32 [B, Hi] (ratio 4) */
    /* outputs (B * n_q entries with speculative verify); out and lse may also be page-locked
       host memory that the device can address (the last kernel then writes them over the
       host link, and the step's completion makes them visible to the host) */
    void* out;                   /* bf16 [B, H, 512] */
    float* lse;                  /* fp32 [B, H], nullable */
    int32_t* sel;                /* int32 [B, k], nullable (ratio 4): the selected candidates as a
                                    set (the same set as csa_topk, -1 padding at the end), in a
                                    fixed order that is not the score order: the same inputs give
                                    the same order and the same output bits */
    /* Optional compression-state ring ([V4-deploy] "ShadowRadix": the state ring nested in the
     * SWA page index; [Day-0] "创新 1 ShadowRadix"): the raw tokens of groups still being
     * filled live in a small per-request ring, token t of request b in row
     * ring_page[b] * ring_size + t % ring_size of ring_pool.  When ring_pool is set, stage 1 reads the pending groups' tokens from the
     * ring instead of kv_raw; the SWA window of stage 4 still reads kv_raw.  The ring must
     * still hold every pending token: n_groups_done[b] * ratio >= n_tokens[b] - ring_size,
     * else the device status gets CSA_ERR_DEVICE_BOUNDS.  Zero-initialise to leave it off. */
    const void* ring_pool;       /* bf16 rows of 1024 B (16-byte aligned), or NULL */
    const int32_t* ring_page;    /* device [B]: request b's ring (0 <= ring_page[b] < ring_n_pages) */
    int32_t ring_size;           /* tokens per ring, a multiple of ratio */
    int64_t ring_n_pages;        /* rings in ring_pool */
    /* Speculative verify ([V4-deploy] "V4 到底改了啥": a one-layer MTP head drafts tokens;
     * "MTP 投機解碼 + 圖內元數據"; 4 draft tokens at bs = 1 in the low-latency setting):
     * n_q query positions per request, 0 or 1 meaning one.  The last n_q
     * of request b's n_tokens[b] tokens are the draft positions; query j sits at token
     * n_tokens[b] - n_q + j and sees the first n_tokens[b] - n_q + j + 1 tokens: the groups
     * completed within them (floor) as candidates, its own top k and its own SWA window.  Stage 1
     * compresses once per request, up to n_tokens[b] / ratio.  q, q_idx, w_h, out, lse and sel
     * then hold B * n_q entries in (request, query) order: q [B, n_q, H, 512] and so on.
     * 1 <= n_q <= 16 and B * n_q <= 65535. */
    int32_t n_q;
    /* HiSparse ([V4-deploy] "HiSparse：把不活躍 KV 甩到 CPU"; [Day-0] "创新 3：HiSparse"): kv_c may be
     * a full mirror of the C4 compressed pool in pinned host memory (kernels read it through its
     * host pointer), with only a working set on the GPU: hs_ws_pool holds hs_n_slots pages of
     * c_page_stride bytes, and hs_ws_table [B, c_page_table_stride] gives the slot of each
     * logical compressed page of each request, or -1.  Stage 4 reads a resident page from its
     * slot and any other straight from the mirror; stage 1 writes new rows to the mirror and, when
     * the page is resident, to its slot.  hs_touch [B, c_page_table_stride], when set, receives
     * hs_step for every compressed page a query read -- the input of the coordinator
     * (csa_hisparse_update), which brings missed pages in between steps.  The index keys stay on
     * the GPU.  Needs ratio 4 and an explicit c_page_table.  Zero-initialise to leave it off. */
    void* hs_ws_pool;            /* device, 16-byte aligned, or NULL */
    int32_t* hs_ws_table;        /* device [B, c_page_table_stride] */
    int64_t hs_n_slots;
    uint32_t* hs_touch;          /* device [B, c_page_table_stride], or NULL */
    uint32_t hs_step;            /* the stamp of this step (>= 1; 0 marks a page never read) */
} csa_decode_params;

/* workspace: device, 16-byte aligned, caller-owned, at least csa_decode_workspace_size(p)
 * bytes; its contents need not start at zero and are overwritten.  The size query returns
 * 0 only when the parameters are rejected (csa_decode then returns the reason). */
csa_status csa_decode(const csa_decode_params* p, void* workspace, size_t ws_bytes, void* stream);
size_t csa_decode_workspace_size(const csa_decode_params* p);

/*
 * csa_decode with stage timing: stage_events (host array of 5 cudaEvent_t, created
 * by the caller with timing enabled) are recorded on `stream` before stage 1 and
 * after stages 1 (compress), 2 (score), 3 (top-k) and 4 (attention + merge).  For
 * ratio 128 the score and top-k events are recorded back to back.  NULL = csa_decode.
 */
csa_status csa_decode_timed(const csa_decode_params* p, void* workspace, size_t ws_bytes, void* stream,
                            void* const* stage_events);

/*
 * csa_decode without a workspace argument, for callers that cannot allocate device
 * memory: code that runs inside an allocator or memory-pool callback, a host that
 * only hands the library its input and output buffers, or a runtime that forbids
 * cudaMalloc once it has started.  (The pages have no counterpart: this is a
 * packaging of csa_decode, not part of the method.)
 * The scratch comes from a fixed 32 MiB array in libcsa's own device memory, which
 * every GPU that loads the library holds until the process exits; a call whose
 * csa_decode_workspace_size() exceeds 32 MiB returns CSA_ERR_WORKSPACE and enqueues
 * nothing.  Nothing is allocated and no scratch contents need to start at zero.
 * The first call on a device looks up the array's device address (with that device
 * current); make that first call before any stream capture.  Every call shares the
 * one array, so calls that overlap on the GPU (other streams, other threads) race.
 */
csa_status csa_decode_noalloc(const csa_decode_params* p, void* stream);

/*
 * Batched copy: up to CSA_COPY_MAX copies enqueued on `stream` as one kernel.  Each copy moves
 * `bytes` bytes from src to dst; either side may be device memory or page-locked host memory
 * allocated with the CUDA runtime (pinned), which with unified virtual addressing the kernel
 * reads and writes through the same pointer.  A decode step's uploads of its new inputs and the
 * download of its outputs are a few small copies; one launch carries them all, where separate
 * copy-engine operations would each add a copy's fixed latency.  src, dst 16-byte aligned,
 * bytes a multiple of 16 (0 allowed), copies not overlapping; otherwise, or for n outside
 * [1, CSA_COPY_MAX], CSA_ERR_INVALID_ARG and nothing is enqueued.  The caller owns the memory.
 * CSA_ERR_CUDA if the launch fails.  Graph capture: yes.
 */
#define CSA_COPY_MAX 16
typedef struct {
    const void* src;
    void* dst;
    uint64_t bytes;
} csa_copy;
csa_status csa_copy_batch(int32_t n, const csa_copy* copies, void* stream);

/* Read and clear the calling device's sticky status word (synchronises `stream`).
 * *out receives a bit set: bit (code-1) for each csa_status code raised on the device. */
csa_status csa_read_device_status(void* stream, int32_t* out);

const char* csa_status_string(csa_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t csa_version(void);

/*
 * Failure-detection self-test: enqueues one kernel that waits on an mbarrier nothing will ever
 * arrive on.  Its wait is bounded the way every wait in the library is (a poll limit with
 * back-off; about a second here, about 8 s for the library's own waits); when it runs out the
 * kernel sets CSA_ERR_TIMEOUT in the device status word (csa_read_device_status) and returns.  Nothing traps or faults, and the
 * context stays usable.  Returns CSA_ERR_CUDA if the launch fails.
 */
csa_status csa_selftest_bounded_wait(void* stream);

/*
 * HiSparse coordinator ([V4-deploy] "HiSparse": a coordinator swaps pages every step and evicts
 * by LRU; [Day-0] "创新 3": a GPU miss is swapped in from the CPU mirror).  A host object holding
 * the working set's bookkeeping: which (request, logical page) each slot holds and the last step
 * that read it.  Its first csa_hisparse_update (or csa_hisparse_collect) allocates a device
 * buffer of 12 * n_slots bytes for the swap plans, freed by csa_hisparse_destroy.
 */
typedef struct csa_hisparse csa_hisparse;
csa_status csa_hisparse_create(int32_t B, int64_t table_stride, int64_t n_slots, csa_hisparse** out);
void csa_hisparse_destroy(csa_hisparse* h);
/* The LRU decision alone, on the host.  touch [B, table_stride] holds the stamps after a step.
 * Every page stamped `step` that is not resident gets a slot, in (request, logical page)
 * order: a free slot (lowest first), else the resident page with the oldest stamp other than
 * `step` (ties: the lowest slot), which is evicted.  When every slot holds a page of this step
 * the rest stay in the mirror.  Writes up to max_plan (request, logical page, slot) triples to
 * plan and the counts; the coordinator's residency table follows the plan. */
csa_status csa_hisparse_plan(csa_hisparse* h, const uint32_t* touch, uint32_t step, int32_t* plan, int64_t max_plan,
                             int64_t* n_in, int64_t* n_evicted);
/* The residency table the coordinator holds: host memory, [B, table_stride] slots or -1. */
const int32_t* csa_hisparse_table(const csa_hisparse* h);
/* After a decode step with p on `stream`: reads p->hs_touch back (waiting for the stream), plans
 * for p->hs_step as csa_hisparse_plan, then enqueues on the stream one gather kernel that copies
 * every planned page from the mirror (kv_c) into its slot, and the new residency table into
 * p->hs_ws_table.  The next step on the stream sees the new working set. */
csa_status csa_hisparse_update(csa_hisparse* h, const csa_decode_params* p, void* stream, int64_t* n_in,
                               int64_t* n_evicted);
/* The same update without stalling the decode stream, in two calls.
 * csa_hisparse_collect, after a decode step with p on `stream`: enqueues the readback of
 *   p->hs_touch into the coordinator's pinned host buffer (no wait); remembers p->hs_step.
 * csa_hisparse_apply, any time later (typically after the next step is enqueued): waits on the
 *   host for that readback only, plans as csa_hisparse_plan for the collected step, then
 *   (1) enqueues on `stream` the residency table with this plan's evictions (the incoming pages
 *   still absent), so that every step enqueued after it reads those pages from the mirror, and
 *   (2) on `side_stream`, once (1) is done: one gather kernel copying the planned pages from the
 *   mirror into their slots, then the table with them installed.  Steps on `stream` overlap (2);
 *   an entry only ever goes from -1 to a slot whose bytes are in place, and no slot is rewritten
 *   before the steps that could read its old page are done.  n_tokens_host [B]: each request's
 *   token count as of the last enqueued step; the page holding a request's newest compressed
 *   row (which the overlapped steps may still write) is not brought in.  An apply waits for the
 *   previous apply's side-stream work before it plans.  The first collect allocates the pinned
 *   buffers (about 12 * B * table_stride + 12 * n_slots bytes) and three events, freed by
 *   csa_hisparse_destroy.  CSA_ERR_INVALID_ARG for an apply without a collect before it. */
csa_status csa_hisparse_collect(csa_hisparse* h, const csa_decode_params* p, void* stream);
csa_status csa_hisparse_apply(csa_hisparse* h, const csa_decode_params* p, const int64_t* n_tokens_host,
                              void* stream, void* side_stream, int64_t* n_in, int64_t* n_evicted);

#ifdef __cplusplus
}
#endif
#endif /* CSA_H_ */
