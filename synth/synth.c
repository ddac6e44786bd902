/*
 * Seeded synthetic input generators shared by the CUDA path's tests/bench and
 * by the CPU oracle's tests.  This file holds NO arithmetic of the attention
 * method: only random draws, their encoding into the storage types the
 * workloads use (bf16, fp8-e4m3, fp32) and integer permutations.
 *
 * Random source: Philox4x32-10, the counter-based generator published by
 * Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3"
 * (SC 2011).  Key = low words of (seed, stream), counter = (block index, high
 * words of seed and stream).  Every
 * element i of a stream depends only on (seed, stream, i), so any sub-range of
 * a tensor can be regenerated on its own and fills run in parallel threads.
 *
 * Normal draws use the Box-Muller transform on pairs of uniforms in (0,1):
 * block b yields elements 4b..4b+3 from its four 32-bit words.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

/* One Philox4x32 block: 10 rounds on counter c[4] under key k[2]. */
void synth_philox4x32_10_raw(const uint32_t c_in[4], const uint32_t k_in[2], uint32_t out[4]) {
    uint32_t c0 = c_in[0], c1 = c_in[1], c2 = c_in[2], c3 = c_in[3];
    uint32_t k0 = k_in[0], k1 = k_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += PHILOX_W0; k1 += PHILOX_W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Block `block` of stream (seed, stream): key = (seed_lo, stream_lo),
 * counter = (block_lo, block_hi, seed_hi, stream_hi). */
static void philox4x32_10(uint64_t block, uint64_t seed, uint64_t stream, uint32_t out[4]) {
    uint32_t c[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)(seed >> 32),
                     (uint32_t)(stream >> 32)};
    uint32_t k[2] = {(uint32_t)seed, (uint32_t)stream};
    synth_philox4x32_10_raw(c, k, out);
}

/* uniform in the open interval (0,1) from a 32-bit word */
static double u01(uint32_t x) { return ((double)x + 0.5) * (1.0 / 4294967296.0); }

static void normals4(uint64_t block, uint64_t seed, uint64_t stream, double z[4]) {
    uint32_t w[4];
    philox4x32_10(block, seed, stream, w);
    const double two_pi = 6.283185307179586476925286766559;
    for (int p = 0; p < 2; ++p) {
        double r = sqrt(-2.0 * log(u01(w[2 * p])));
        double t = two_pi * u01(w[2 * p + 1]);
        z[2 * p] = r * cos(t);
        z[2 * p + 1] = r * sin(t);
    }
}

/* float -> bf16 bits, round to nearest even (inputs are finite) */
static uint16_t enc_bf16(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7FFFu + lsb;
    return (uint16_t)(b >> 16);
}

/* double -> fp8 e4m3 (OCP "E4M3FN": bias 7, no inf, max 448), round to
 * nearest even, saturating to +-448. */
static uint8_t enc_e4m3(double x) {
    uint8_t s = (x < 0) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return s | 0x7E;
    if (a == 0.0) return s;
    int e;
    frexp(a, &e);           /* a = m * 2^e, m in [0.5,1) -> floor(log2 a) = e-1 */
    int fl = e - 1;
    double q;
    if (fl < -6) {          /* subnormal grid: 2^-9 */
        q = nearbyint(ldexp(a, 9));
        if (q >= 8.0) return s | 0x08;          /* rounded up to 2^-6 */
        return s | (uint8_t)q;
    }
    q = nearbyint(ldexp(a, 3 - fl));            /* in [8,16] */
    if (q >= 16.0) { q = 8.0; fl += 1; }
    if (fl > 8 || (fl == 8 && q > 14.0)) return s | 0x7E;
    return s | (uint8_t)(((fl + 7) << 3) | ((int)q - 8));
}

/* ------------------------------------------------------------------ fills */

enum { K_NORMAL_BF16 = 0, K_NORMAL_F32 = 1, K_NORMAL_E4M3 = 2, K_UNIFORM_F32 = 3 };

typedef struct {
    int kind;
    void* out;
    int64_t begin, end;     /* element range [begin,end) of the stream to write */
    int64_t out_offset;     /* element index in `out` of stream element `begin` */
    uint64_t seed, stream;
    double a, b;            /* normal: mean, std; uniform: lo, hi */
} fill_job;

static void* fill_worker(void* arg) {
    fill_job* j = (fill_job*)arg;
    int64_t i = j->begin;
    while (i < j->end) {
        uint64_t blk = (uint64_t)i >> 2;
        double z[4];
        if (j->kind == K_UNIFORM_F32) {
            uint32_t w[4];
            philox4x32_10(blk, j->seed, j->stream, w);
            for (int t = 0; t < 4; ++t) z[t] = j->a + (j->b - j->a) * u01(w[t]);
        } else {
            normals4(blk, j->seed, j->stream, z);
            for (int t = 0; t < 4; ++t) z[t] = j->a + j->b * z[t];
        }
        for (int t = (int)(i & 3); t < 4 && i < j->end; ++t, ++i) {
            int64_t o = j->out_offset + (i - j->begin);
            switch (j->kind) {
                case K_NORMAL_BF16: ((uint16_t*)j->out)[o] = enc_bf16((float)z[t]); break;
                case K_NORMAL_E4M3: ((uint8_t*)j->out)[o] = enc_e4m3(z[t]); break;
                default: ((float*)j->out)[o] = (float)z[t]; break;
            }
        }
    }
    return NULL;
}

static void run_fill(int kind, void* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream,
                     double a, double b, int nthreads) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if (n < (1 << 16)) nthreads = 1;
    fill_job jobs[64];
    pthread_t th[64];
    int64_t per = (n + nthreads - 1) / nthreads;
    per = (per + 3) & ~(int64_t)3;
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t lo = begin + (int64_t)t * per;
        int64_t hi = lo + per;
        if (hi > begin + n) hi = begin + n;
        if (lo >= hi) break;
        jobs[t] = (fill_job){kind, out, lo, hi, lo - begin, seed, stream, a, b};
        used++;
    }
    for (int t = 1; t < used; ++t) pthread_create(&th[t], NULL, fill_worker, &jobs[t]);
    fill_worker(&jobs[0]);
    for (int t = 1; t < used; ++t) pthread_join(th[t], NULL);
}

void synth_normal_bf16(uint16_t* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream,
                       double mean, double std, int nthreads) {
    run_fill(K_NORMAL_BF16, out, begin, n, seed, stream, mean, std, nthreads);
}
void synth_normal_f32(float* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream,
                      double mean, double std, int nthreads) {
    run_fill(K_NORMAL_F32, out, begin, n, seed, stream, mean, std, nthreads);
}
void synth_normal_e4m3(uint8_t* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream,
                       double mean, double std, int nthreads) {
    run_fill(K_NORMAL_E4M3, out, begin, n, seed, stream, mean, std, nthreads);
}
void synth_uniform_f32(float* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream,
                       double lo, double hi, int nthreads) {
    run_fill(K_UNIFORM_F32, out, begin, n, seed, stream, lo, hi, nthreads);
}

/* raw 32-bit words of a stream: element i is word (i & 3) of block i >> 2 */
void synth_u32(uint32_t* out, int64_t begin, int64_t n, uint64_t seed, uint64_t stream) {
    for (int64_t i = begin; i < begin + n; ++i) {
        uint32_t w[4];
        philox4x32_10((uint64_t)i >> 2, seed, stream, w);
        out[i - begin] = w[i & 3];
    }
}

/* uniform integer in [0, m) from element i of a stream (64-bit multiply-shift) */
static uint32_t uniform_below(uint64_t i, uint64_t seed, uint64_t stream, uint32_t m) {
    uint32_t w[4];
    philox4x32_10(i, seed, stream, w);
    uint64_t x = ((uint64_t)w[0] << 32) | w[1];
    return (uint32_t)(((unsigned __int128)x * m) >> 64);
}

/* Fisher-Yates permutation of 0..n-1: draw i uses block i of the stream */
void synth_permutation(int32_t* out, int64_t n, uint64_t seed, uint64_t stream) {
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; --i) {
        int64_t j = uniform_below((uint64_t)i, seed, stream, (uint32_t)(i + 1));
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}

/* n integers uniform in [lo, hi] (inclusive) */
void synth_uniform_int(int64_t* out, int64_t n, int64_t lo, int64_t hi, uint64_t seed, uint64_t stream) {
    uint32_t m = (uint32_t)(hi - lo + 1);
    for (int64_t i = 0; i < n; ++i) out[i] = lo + uniform_below((uint64_t)i, seed, stream, m);
}

/* Scatter logical rows into a paged pool: logical row r (page r / rpp, slot
 * r % rpp) goes to physical page page_table[r / rpp].  Pure data movement. */
void synth_scatter_pages(const uint8_t* logical, int64_t n_rows, int64_t row_bytes, int32_t rpp,
                         const int32_t* page_table, int64_t page_stride_bytes, uint8_t* pool) {
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t p = page_table[r / rpp];
        memcpy(pool + p * page_stride_bytes + (r % rpp) * row_bytes, logical + r * row_bytes,
               (size_t)row_bytes);
    }
}

/* Inverse of synth_scatter_pages. */
void synth_gather_pages(const uint8_t* pool, int64_t n_rows, int64_t row_bytes, int32_t rpp,
                        const int32_t* page_table, int64_t page_stride_bytes, uint8_t* logical) {
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t p = page_table[r / rpp];
        memcpy(logical + r * row_bytes, pool + p * page_stride_bytes + (r % rpp) * row_bytes,
               (size_t)row_bytes);
    }
}
