/*
 * CPU ORACLE for the C4 hybrid-sparse-attention decode step.
 *
 * Test infrastructure only: tests, the smoke check and the benchmark's CPU
 * baseline call it; the product path never does.  Plain single-threaded C,
 * compiled with -O2 -ffp-contract=off (no fused operations except the fmaf
 * calls written out below).  It shares no code with the CUDA path.
 *
 * Sources (web pages; quoted by title and section):
 *   [V4-deploy]  "DeepSeek-V4 本地部署，SGLang 把活做絕了"
 *                 sec. "V4 到底改了啥" (hybrid attention: every layer = SWA of the
 *                 last 128 raw tokens + C4 (4:1 compression, top-512 sparse) or
 *                 C128 (128:1 compression, dense));
 *                 sec. "Kernel 層一堆狠活" (one call for SWA + extra attention;
 *                 Flash Compressor; Lightning TopK: 256K candidates -> top-512).
 *   [Day-0]      "SGLang 如何为 DeepSeek V4 打造「Day-0」推理加速"
 *                 sec. "创新 2：Flash Compressor + Lightning TopK" (the five-stage
 *                 compression chain load -> score -> softmax -> weighted sum ->
 *                 store; radix select of the top K = 512 with a threshold).
 * Where the pages leave the arithmetic open, the problem statement fixes it:
 *   gate s_i = kv_i . w_gate + b_pos[i];  index score[g] = sum_h w_h *
 *   ReLU(q_idx[h] . k_idx[g]) in fp32 in a fixed chunk order; top-k by
 *   descending score, ties to the lower index.
 *
 * Parity status of each function is stated beside it ("pinned by" lists the
 * independent checks in tests/test_oracle_pins.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_LATENT 512
#define D_INDEX 128

/* ---------------------------------------------------------------------------
 * Storage types, decoded from their definitions.
 *   bf16: the upper 16 bits of an IEEE-754 binary32.
 *   e4m3 (OCP 8-bit floating point, E4M3FN): 1 sign, 4 exponent bits (bias 7),
 *   3 mantissa bits; exponent 0 = subnormal (m * 2^-9); S.1111.111 = NaN.
 * Pinned by: every code compared with torch's bfloat16 / float8_e4m3fn casts.
 * ------------------------------------------------------------------------- */
float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

float orc_e4m3_to_f32(uint8_t b) {
    int s = b >> 7, e = (b >> 3) & 0xF, m = b & 7;
    float v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0)
        v = ldexpf((float)m, -9);
    else
        v = ldexpf((float)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* Round a double to the nearest bf16 (ties to even) in ONE rounding step.
 * bf16 keeps 8 significant bits; normal exponents -126..127; subnormal spacing
 * 2^-133.  Pinned by: brute-force nearest-neighbour search in exact rationals. */
uint16_t orc_f64_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);
    int fl = e - 1; /* floor(log2 a) */
    double v;
    if (fl < -126) {
        v = ldexp(nearbyint(ldexp(a, 133)), -133);
    } else {
        v = ldexp(nearbyint(ldexp(a, 7 - fl)), fl - 7);
    }
    if (v >= 0x1p128) return sign | 0x7F80; /* overflow to infinity */
    float f = (float)v;                      /* exact: v is on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, 4);
    return sign | (uint16_t)(u >> 16);
}

/* ---------------------------------------------------------------------------
 * Stage 1: softmax-gated r:1 compression ([V4-deploy] "V4 到底改了啥": C4 = 4:1,
 * C128 = 128:1; [Day-0] "创新 2": score -> softmax -> weighted sum per group).
 * Group j covers raw tokens r*j .. r*j+r-1 (disjoint groups from token 0):
 *   s_i = sum_d x_{rj+i}[d] * w_gate[d] + b_pos[i]
 *   a   = softmax(s)            (max-subtracted)
 *   c_j = sum_i a_i * x_{rj+i}  -> bf16 (one rounding)
 * All arithmetic in fp64.
 * Pinned by: identical tokens -> that token; sum a = 1; w_gate = b_pos = 0 ->
 * arithmetic mean; one-hot b_pos -> that token; permutation of (tokens, b_pos)
 * inside a group; hand-computed golden group.
 * x: bf16 [n_tokens, 512] in logical token order.
 * out_bf16 [n_groups, 512]; out_f64 [n_groups, 512] and gates [n_groups, r]
 * are optional (unrounded results).
 * ------------------------------------------------------------------------- */
int orc_compress(const uint16_t* x, int64_t n_tokens, int ratio, const float* w_gate, const float* b_pos,
                 int64_t first_group, int64_t n_groups, uint16_t* out_bf16, double* out_f64, double* gates) {
    if (ratio <= 0 || ratio > 4096) return 1;
    if (first_group < 0 || n_groups < 0 || (first_group + n_groups) * ratio > n_tokens) return 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)ratio);
    double c[D_LATENT];
    for (int64_t g = 0; g < n_groups; ++g) {
        const int64_t j = first_group + g;
        const uint16_t* xg = x + j * ratio * D_LATENT;
        double mx = -INFINITY;
        for (int i = 0; i < ratio; ++i) {
            double acc = 0.0;
            for (int d = 0; d < D_LATENT; ++d)
                acc += (double)orc_bf16_to_f32(xg[i * D_LATENT + d]) * (double)w_gate[d];
            s[i] = acc + (double)b_pos[i];
            if (s[i] > mx) mx = s[i];
        }
        double z = 0.0;
        for (int i = 0; i < ratio; ++i) {
            s[i] = exp(s[i] - mx);
            z += s[i];
        }
        for (int i = 0; i < ratio; ++i) s[i] /= z; /* s now holds the gate weights a_i */
        if (gates)
            for (int i = 0; i < ratio; ++i) gates[g * ratio + i] = s[i];
        for (int d = 0; d < D_LATENT; ++d) c[d] = 0.0;
        for (int i = 0; i < ratio; ++i)
            for (int d = 0; d < D_LATENT; ++d) c[d] += s[i] * (double)orc_bf16_to_f32(xg[i * D_LATENT + d]);
        for (int d = 0; d < D_LATENT; ++d) {
            if (out_bf16) out_bf16[g * D_LATENT + d] = orc_f64_to_bf16(c[d]);
            if (out_f64) out_f64[g * D_LATENT + d] = c[d];
        }
    }
    free(s);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Stage 2: indexer score over every compressed candidate ([V4-deploy] "Kernel
 * 層一堆狠活": the indexer picks top-512 of 256K candidates at 1M context).
 *   score[g] = sum_h w_h * ReLU(q_idx[h] . k_idx[g])
 * fp32, fixed order (bit-exact contract shared with the GPU):
 *   chain j = dims 32j..32j+31 (j = 0..3):  Q[j] = q[32j]*k[32j];
 *                                         Q[j] = fmaf(q[32j+i], k[32j+i], Q[j]) for i = 1..31
 *   dot_h = (Q[0] + Q[2]) + (Q[1] + Q[3])
 *   acc = 0;  acc = fmaf(w_h, ReLU(dot_h), acc) for h = 0..Hi-1, ReLU(x) = x > 0 ? x : +0
 * q_idx bf16 [Hi,128]; k_idx bf16 or e4m3 [G,128] (logical row order).
 * Pinned by: exact small-integer cases; fp64 error bound for Hi = 1; ReLU of
 * all-negative dots; exact doubling under w -> 2w; hand-computed golden case
 * in which the chain order decides the rounding.
 * ------------------------------------------------------------------------- */
void orc_index_score(const uint16_t* q_idx, const float* w_h, int Hi, const void* k_idx, int k_fp8, int64_t G,
                     float* scores) {
    float q[64][D_INDEX];
    for (int h = 0; h < Hi && h < 64; ++h)
        for (int d = 0; d < D_INDEX; ++d) q[h][d] = orc_bf16_to_f32(q_idx[h * D_INDEX + d]);
    for (int64_t g = 0; g < G; ++g) {
        float k[D_INDEX];
        for (int d = 0; d < D_INDEX; ++d)
            k[d] = k_fp8 ? orc_e4m3_to_f32(((const uint8_t*)k_idx)[g * D_INDEX + d])
                         : orc_bf16_to_f32(((const uint16_t*)k_idx)[g * D_INDEX + d]);
        float acc = 0.0f;
        for (int h = 0; h < Hi; ++h) {
            float Q[4];
            for (int j = 0; j < 4; ++j) {
                float p = q[h][32 * j] * k[32 * j];
                for (int i = 1; i < 32; ++i) p = fmaf(q[h][32 * j + i], k[32 * j + i], p);
                Q[j] = p;
            }
            float dot = (Q[0] + Q[2]) + (Q[1] + Q[3]);
            float r = dot > 0.0f ? dot : 0.0f;
            acc = fmaf(w_h[h], r, acc);
        }
        scores[g] = acc;
    }
}

/* ---------------------------------------------------------------------------
 * Stage 3: top-k selection ([Day-0] "创新 2": Lightning TopK keeps the K = 512
 * best candidates; the problem statement fixes the order: descending score,
 * ties to the lower index).  Defined as a full sort under a total order:
 *   key(x) = order-preserving 32-bit image of the fp32 score (-0 == +0):
 *            negative -> ~bits, non-negative -> bits | 0x80000000
 *   sort by (key desc, index asc); output the first min(k, G) indices, then -1.
 * Pinned by: Python's sorted() on (-score, index) with planted ties, +-0,
 * negatives and infinities; k >= G.
 * ------------------------------------------------------------------------- */
uint32_t orc_score_key(float s) {
    uint32_t u;
    memcpy(&u, &s, 4);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

typedef struct {
    uint32_t key;
    int32_t idx;
} orc_kv;

static int orc_kv_cmp(const void* a, const void* b) {
    const orc_kv* x = (const orc_kv*)a;
    const orc_kv* y = (const orc_kv*)b;
    if (x->key != y->key) return x->key > y->key ? -1 : 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

static void orc_kv_swap(orc_kv* x, orc_kv* y) {
    const orc_kv t = *x;
    *x = *y;
    *y = t;
}

/* Rearrange a[0..n) so that a[m] holds the element a full sort would put there, everything
 * before it precedes it in the order and everything after follows it (selection by
 * repeated partitioning, pivot = median of the first, middle and last element).  The keys
 * are distinct under the total order, so the partition is well defined. */
static void orc_select_nth(orc_kv* a, int64_t n, int64_t m) {
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (orc_kv_cmp(&a[mid], &a[lo]) < 0) orc_kv_swap(&a[mid], &a[lo]);
        if (orc_kv_cmp(&a[hi], &a[lo]) < 0) orc_kv_swap(&a[hi], &a[lo]);
        if (orc_kv_cmp(&a[hi], &a[mid]) < 0) orc_kv_swap(&a[hi], &a[mid]);
        const orc_kv p = a[mid];
        int64_t i = lo, j = hi;
        while (i <= j) {
            while (orc_kv_cmp(&a[i], &p) < 0) ++i;
            while (orc_kv_cmp(&p, &a[j]) < 0) --j;
            if (i <= j) {
                orc_kv_swap(&a[i], &a[j]);
                ++i;
                --j;
            }
        }
        if (m <= j)
            hi = j;
        else if (m >= i)
            lo = i;
        else
            break; /* a[m] equals the pivot: in place */
    }
}

/* Top-k as in orc_topk, by selection: the k first elements by the same total order are
 * moved to the front (orc_select_nth on rank k - 1), and only those k are sorted.  The
 * result is the same (the order is total, so the k best and their order are unique); it is
 * the second CPU method the timing reports. */
int orc_topk_select(const float* scores, int64_t G, int k, int32_t* idx_out, uint32_t* keys_out) {
    if (G < 0 || k < 0) return 1;
    orc_kv* a = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)(G > 0 ? G : 1));
    if (!a) return 2;
    for (int64_t g = 0; g < G; ++g) {
        a[g].key = orc_score_key(scores[g]);
        a[g].idx = (int32_t)g;
    }
    const int64_t m = k < G ? k : G;
    if (m > 0 && m < G) orc_select_nth(a, G, m - 1);
    qsort(a, (size_t)m, sizeof(orc_kv), orc_kv_cmp);
    for (int i = 0; i < k; ++i) {
        idx_out[i] = i < G ? a[i].idx : -1;
        if (keys_out) keys_out[i] = i < G ? a[i].key : 0u;
    }
    free(a);
    return 0;
}

int orc_topk(const float* scores, int64_t G, int k, int32_t* idx_out, uint32_t* keys_out) {
    if (G < 0 || k < 0) return 1;
    orc_kv* a = (orc_kv*)malloc(sizeof(orc_kv) * (size_t)(G > 0 ? G : 1));
    if (!a) return 2;
    for (int64_t g = 0; g < G; ++g) {
        a[g].key = orc_score_key(scores[g]);
        a[g].idx = (int32_t)g;
    }
    qsort(a, (size_t)G, sizeof(orc_kv), orc_kv_cmp); /* total order: the result is unique */
    for (int i = 0; i < k; ++i) {
        idx_out[i] = i < G ? a[i].idx : -1;
        if (keys_out) keys_out[i] = i < G ? a[i].key : 0u;
    }
    free(a);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Stage 4: one attention over a set of latent rows under a single softmax
 * ([V4-deploy] "Kernel 層一堆狠活": SWA and the extra C4/C128 attention in one
 * call).  K = V = the bf16 latent row (512 dims).  For head h:
 *   l_j = scale * sum_d q[h][d] * K_j[d];  p = softmax(l);  o_h = sum_j p_j V_j
 *   lse_h = log sum_j exp(l_j)
 * fp64; o rounded once to bf16.
 * Pinned by: one key -> its row; q = 0 -> mean of rows and lse = log n;
 * numpy float64 textbook softmax attention on random sets.
 * rows: bf16 [n_keys, 512].
 * ------------------------------------------------------------------------- */
void orc_attention(const uint16_t* q, int H, float scale, const uint16_t* rows, int64_t n_keys, uint16_t* out_bf16,
                   double* out_f64, double* lse) {
    double* l = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
    double o[D_LATENT];
    for (int h = 0; h < H; ++h) {
        const uint16_t* qh = q + (int64_t)h * D_LATENT;
        double mx = -INFINITY;
        for (int64_t j = 0; j < n_keys; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D_LATENT; ++d)
                acc += (double)orc_bf16_to_f32(qh[d]) * (double)orc_bf16_to_f32(rows[j * D_LATENT + d]);
            l[j] = (double)scale * acc;
            if (l[j] > mx) mx = l[j];
        }
        double z = 0.0;
        for (int d = 0; d < D_LATENT; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < n_keys; ++j) {
            double p = exp(l[j] - mx);
            z += p;
            for (int d = 0; d < D_LATENT; ++d) o[d] += p * (double)orc_bf16_to_f32(rows[j * D_LATENT + d]);
        }
        for (int d = 0; d < D_LATENT; ++d) {
            double v = n_keys > 0 ? o[d] / z : 0.0;
            if (out_bf16) out_bf16[(int64_t)h * D_LATENT + d] = orc_f64_to_bf16(v);
            if (out_f64) out_f64[(int64_t)h * D_LATENT + d] = v;
        }
        if (lse) lse[h] = n_keys > 0 ? mx + log(z) : -INFINITY;
    }
    free(l);
}

/* Key set of the sparse + SWA attention: the selected compressed entries (any
 * order; -1 entries are padding and skipped), then the last W = min(swa, N)
 * raw tokens.  No de-duplication between the two sets. */
int orc_sparse_attn(const uint16_t* q, int H, float scale, const uint16_t* cpool, int64_t G, const int32_t* sel,
                    int n_sel, const uint16_t* raw, int64_t n_tokens, int swa, uint16_t* out_bf16, double* out_f64,
                    double* lse) {
    int64_t W = swa < n_tokens ? swa : n_tokens;
    if (W < 0) W = 0;
    uint16_t* rows = (uint16_t*)malloc(sizeof(uint16_t) * D_LATENT * (size_t)(n_sel + W + 1));
    if (!rows) return 2;
    int64_t n = 0;
    for (int i = 0; i < n_sel; ++i) {
        if (sel[i] < 0) continue;
        if (sel[i] >= G) {
            free(rows);
            return 1;
        }
        memcpy(rows + n * D_LATENT, cpool + (int64_t)sel[i] * D_LATENT, D_LATENT * sizeof(uint16_t));
        ++n;
    }
    for (int64_t t = n_tokens - W; t < n_tokens; ++t) {
        memcpy(rows + n * D_LATENT, raw + t * D_LATENT, D_LATENT * sizeof(uint16_t));
        ++n;
    }
    orc_attention(q, H, scale, rows, n, out_bf16, out_f64, lse);
    free(rows);
    return 0;
}

/* ---------------------------------------------------------------------------
 * The decode step of one request: stage 1 on the completed groups that are
 * not yet in the pool ([n_groups_done, N/r)), written into cpool as bf16;
 * then for C4 (dense == 0) stage 2 over all G = N/r candidates, stage 3
 * (top-k) and stage 4 over the selection + SWA; for C128 (dense != 0) stage 4
 * over all G entries + SWA ([V4-deploy] "V4 到底改了啥": C128 is attended densely).
 * cpool: bf16 [G, 512], rows < n_groups_done are inputs, the rest outputs.
 * sel [k] and scores [G] are optional outputs.
 * ------------------------------------------------------------------------- */
int orc_decode_request(const uint16_t* raw, int64_t n_tokens, uint16_t* cpool, int64_t n_groups_done, int ratio,
                       int dense, const float* w_gate, const float* b_pos, const uint16_t* q_idx, const float* w_h,
                       int Hi, const void* k_idx, int k_fp8, int k, const uint16_t* q, int H, float scale, int swa,
                       uint16_t* out_bf16, double* out_f64, double* lse, int32_t* sel, float* scores) {
    /* the candidates are the groups completed within the n_tokens tokens (floor); the tokens of
       a trailing partial group take part only through the SWA window */
    if (ratio <= 0 || n_tokens < 0) return 1;
    const int64_t G = n_tokens / ratio;
    if (n_groups_done < 0 || n_groups_done > G) return 1;
    int rc = orc_compress(raw, n_tokens, ratio, w_gate, b_pos, n_groups_done, G - n_groups_done,
                          cpool + n_groups_done * D_LATENT, NULL, NULL);
    if (rc) return rc;
    if (dense) {
        int32_t* all = (int32_t*)malloc(sizeof(int32_t) * (size_t)(G > 0 ? G : 1));
        for (int64_t g = 0; g < G; ++g) all[g] = (int32_t)g;
        rc = orc_sparse_attn(q, H, scale, cpool, G, all, (int)G, raw, n_tokens, swa, out_bf16, out_f64, lse);
        free(all);
        return rc;
    }
    float* s = scores ? scores : (float*)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
    int32_t* idx = sel ? sel : (int32_t*)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    orc_index_score(q_idx, w_h, Hi, k_idx, k_fp8, G, s);
    rc = orc_topk(s, G, k, idx, NULL);
    if (!rc) rc = orc_sparse_attn(q, H, scale, cpool, G, idx, k, raw, n_tokens, swa, out_bf16, out_f64, lse);
    if (!scores) free(s);
    if (!sel) free(idx);
    return rc;
}
