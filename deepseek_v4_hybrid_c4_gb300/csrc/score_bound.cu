// Stage 2 on the tensor cores: a bracket around every candidate's fixed-order index score
// ("DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "Kernel 層一堆狠活": the indexer over 256K
// candidates feeds the top-512; the indexer's q.k products are a dense contraction).
//
// The top-k ranks the fixed-order fp32 score s of score.cu (four 32-long fma chains per head).
// Here the dots run as one tcgen05 MMA per tile of 128 candidates: D[g][n] = sum_j K[g][j] Q[n][j]
// with bf16 operands in shared memory and fp32 accumulators in tensor memory, n over every
// (query position p, head h) of the request (column p * HI + h).  From them
//   s~ = sum_h w_h ReLU(D[g][p HI + h])                      (fp32, heads in order)
//   e  = 2^-13 max_j |k_gj| sum_h |w_h| ||q_h||_1 + 1e-30    (rounded up)
// and |s~ - s| <= e: with d_h the exact dot and S_h = sum_j |q_hj k_gj| <= ||q_h||_1 max_j |k_gj|,
//   |s~ - s| <= sum_h |w_h| (|D - d_h| + |d_h - fp32 chains|) + the two weighted sums' roundings.
// bf16 products are exact in fp32, so the chains of 32 fmas and the two additions err by at
// most 33 * 2^-24 S_h; the MMA's fp32 accumulation is taken to err by at most 2^-14 S_h (IEEE
// summation of 128 terms in any order errs by at most 127 * 2^-24 S_h: a margin of about 500);
// the weighted sums add at most 2^-20 sum_h |w_h| S_h.  The sum stays below 2^-13 sum |w_h| S_h;
// the 1e-30 covers products that leave the normal range.  A non-finite dot, key or bound, or a
// bound past 1e30, gives the bracket (-inf, +inf); a row whose page id is out of range gets
// [0, 0] (the fixed-order kernel writes 0 for it) and CSA_ERR_DEVICE_BOUNDS.
//
// Output: upper = s~ + e (rounded up) per candidate and, when asked, lower = s~ - e (rounded
// down); with hist, a histogram of the top HB bits of the lower bounds' keys per batch entry
// (HB = 14 for one query position per request, 13 for two, 12 for three or four): the bin
// holding the k-th largest lower bound is a threshold that at least k exact scores reach, and
// every candidate whose upper bound stays below it is out.
//
// CTA: one per SM, 6 warps, over a contiguous share of the batch's tiles.  Warp 0 looks up
// the pages of four tiles at a time, one window ahead, and issues the TMA copies (16-row x
// 128-byte boxes, 128-byte swizzle, K-major) into a ring of up to 6 stages.  Warp 1 stages the
// request's query as the MMA's B operand (zero rows past Hi per position) and issues the
// MMAs, two accumulator buffers in tensor memory.  Warps 2..5 each read their TMEM lane
// quarter (one candidate per thread), take max |k| of the candidate's row from the stage and
// write the bracket.
#include <cuda.h>

#include <cfloat>

#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int SB_ROWS = 128;                   // candidates per tile (MMA M)
constexpr int SB_UNIT = 16;                    // rows per TMA box
constexpr uint32_t SB_HALF = SB_ROWS * 128;    // dims 0..63 (or 64..127) of a tile: 16 KB
constexpr uint32_t SB_TILE = 2 * SB_HALF;
constexpr int SB_EPI = 8;                      // epilogue warps: two groups of four, one per accumulator buffer
constexpr int SB_THREADS = (2 + SB_EPI) * 32;
constexpr int SB_NQ = 4;                       // query positions per request, at most
constexpr int SB_MAX_STAGES = 6;
constexpr int SB_FLUSH_T = SB_EPI * 32;         // epilogue threads
constexpr float SB_MARGIN = 1.220703125e-4f;   // 2^-13
constexpr int64_t SB_PAST = INT64_MIN;         // a unit with nothing to copy

struct BoundArgs {
    const uint16_t* q_idx;   // [B * nq][Hi][128]
    const float* w_h;        // [B * nq][Hi]
    int Hi, nq, N;           // N: MMA width, nq * HI rounded up to 16
    const int32_t* pt;
    int64_t pt_stride, n_pages;
    int32_t rpp;
    float* upper;            // [B * nq] rows score_stride apart
    float* lower;            // the same, or nullptr
    int64_t score_stride;
    int B;                   // requests
    const int64_t* n_tokens; // decode mode; nullptr: one request of G candidates
    int ratio;
    int64_t G;
    uint32_t* hist;          // [B * nq][kHistBlock] (zeroed by the preceding kernel) or nullptr
    int hb;                  // histogram bits (bins 2^hb per batch entry)
    int32_t* status;
    int S;                   // ring stages
};

struct BoundLayout {
    uint32_t q, hist, cst, bar, tmem, total;
};
__host__ __device__ inline BoundLayout bound_layout(int S, int N, int nq, bool hist, int hb) {
    BoundLayout L;
    uint32_t o = (uint32_t)S * SB_TILE;
    L.q = o;
    o += (uint32_t)N * 256u;
    L.hist = o;
    o += hist ? ((uint32_t)nq << hb) * 4u : 0u;
    L.cst = o;
    o += SB_EPI * 512;  // per epilogue warp: weights [SB_NQ * 16], bounds [SB_NQ], lengths [SB_NQ]
    L.bar = o;
    o += 256;
    L.tmem = o;
    o += 16;
    L.total = o + 1024;  // alignment slack
    return L;
}

// Request r's candidates: the largest count over its query positions (the last one's).
struct TileCursor {
    int r = -1;
    int64_t base = 0, tiles = 0, G = 0;
    __device__ void load(const BoundArgs& a) {
        G = a.n_tokens ? query_tokens(a.n_tokens, r * a.nq + a.nq - 1, a.nq) / a.ratio : a.G;
        if (G < 0) G = 0;
        tiles = (G + SB_ROWS - 1) / SB_ROWS;
    }
    __device__ bool seek(const BoundArgs& a, int64_t m) {
        if (r < 0) {
            if (a.B <= 0) return false;
            r = 0;
            load(a);
        }
        if (r >= a.B) return false;
        while (m >= base + tiles) {
            base += tiles;
            if (++r >= a.B) return false;
            load(a);
        }
        return true;
    }
};

// Sum of |x| over the 8 bf16 values of a 16-byte chunk.
__device__ __forceinline__ float abs_sum8(uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) s += fabsf(bf16lo(w[i])) + fabsf(bf16hi(w[i]));
    return s;
}

template <int HI>
__global__ void __launch_bounds__(SB_THREADS, 1)
    score_bound_kernel(const __grid_constant__ CUtensorMap kmap, BoundArgs a) {
    constexpr int NT = SB_NQ * HI;                       // accumulator columns per buffer (>= N)
    constexpr uint32_t TCOLS = 2 * NT < 32 ? 32 : 2 * NT;  // a power of two
    extern __shared__ __align__(1024) uint8_t sb_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sb_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const BoundLayout L = bound_layout(a.S, a.N, a.nq, a.hist != nullptr, a.hb);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.S;
    const uint32_t bar = sbase + L.bar;
    // barriers: full[S] (+0), empty[S] (+48), acc full[2] (+96), acc empty[2] (+112),
    // query free (+128), epilogue rendezvous (+136); unit masks [S] (+160)
    const uint32_t accfull = bar + 96, accempty = bar + 112, qbar = bar + 128, ebar = bar + 136;
    uint32_t* umask = reinterpret_cast<uint32_t*>(sm + L.bar + 160);
    uint32_t* hist = reinterpret_cast<uint32_t*>(sm + L.hist);

    pdl_launch_dependents();  // the select may be scheduled now; it waits for this grid to finish
    __shared__ int64_t s_tot[SB_THREADS / 32];
    int64_t t = 0;
    for (int r = threadIdx.x; r < a.B; r += SB_THREADS) {
        int64_t G = a.n_tokens ? query_tokens(a.n_tokens, r * a.nq + a.nq - 1, a.nq) / a.ratio : a.G;
        if (G < 0) G = 0;
        t += (G + SB_ROWS - 1) / SB_ROWS;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s_tot[warp] = t;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar + 8u * s, 1);           // the producer's arrive + the copies' bytes
            mbar_init(bar + 48u + 8u * s, 5);     // the MMAs' commit + the tile's 4 epilogue warps
        }
        mbar_init(accfull, 1);
        mbar_init(accfull + 8, 1);
        mbar_init(accempty, 4);
        mbar_init(accempty + 8, 4);
        mbar_init(qbar, 1);
        mbar_init(ebar, SB_EPI);
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    }
    if (a.hist)
        for (int i = threadIdx.x; i < (a.nq << a.hb) / 4; i += SB_THREADS)
            st_shared_zero16(smem_u32(hist) + 16u * (uint32_t)i);
    if (warp == 1) {
        tmem_alloc(sbase + L.tmem, TCOLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int64_t total = 0;
#pragma unroll
    for (int w = 0; w < SB_THREADS / 32; ++w) total += s_tot[w];
    const int64_t m0 = (int64_t)blockIdx.x * total / gridDim.x;
    const int64_t nk = ((int64_t)blockIdx.x + 1) * total / gridDim.x - m0;
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + L.tmem);

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        // Lane 8w + u looks up unit u of tile 4i + w of window i; two register sets
        // alternate (even / odd windows), the next window looked up as the current one starts.
        TileCursor lc;
        int64_t pp0 = SB_PAST, pp1 = SB_PAST;
        int sl0 = 0, sl1 = 0;
        auto look = [&](int64_t wi, int64_t& pp, int& sl) {
            pp = SB_PAST;
            sl = 0;
            const int64_t jl = wi * 4 + (lane >> 3);
            if (jl < nk && lc.seek(a, m0 + jl)) {
                const int64_t row0 = (m0 + jl - lc.base) * SB_ROWS + (int64_t)(lane & 7) * SB_UNIT;
                if (row0 < lc.G) {
                    const int64_t lp = row0 / a.rpp;
                    sl = (int)(row0 - lp * a.rpp);
                    pp = a.pt ? (int64_t)__ldg(a.pt + (int64_t)lc.r * a.pt_stride + lp) : lp;
                }
            }
        };
        look(0, pp0, sl0);
        look(1, pp1, sl1);
        int64_t issued = 0;
        for (int64_t jl = 0; jl < nk; ++jl) {
            if ((jl & 3) == 0 && jl > 0) {  // window jl/4 starts: the set of window jl/4 - 1 is free
                if ((jl >> 2) & 1) look(jl / 4 + 1, pp0, sl0);
                else look(jl / 4 + 1, pp1, sl1);
            }
            const int s = (int)(jl % S);
            if (jl >= S && !mbar_wait(bar + 48u + 8u * s, (uint32_t)(((jl / S) & 1) ^ 1))) {
                raise_status(a.status, CSA_ERR_TIMEOUT);
                break;
            }
            const bool odd = (jl >> 2) & 1;
            const int64_t pp = odd ? pp1 : pp0;
            const int sl = odd ? sl1 : sl0;
            const bool mine = (lane >> 3) == (int)(jl & 3);
            const bool valid = mine && pp != SB_PAST && pp >= 0 && pp < a.n_pages;
            if (mine && pp != SB_PAST && !valid) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
            const uint32_t units = (__ballot_sync(0xffffffffu, valid) >> (8 * (jl & 3))) & 0xFFu;
            if (lane == 0) {
                umask[s] = units;
                mbar_arrive_expect_tx(bar + 8u * s, (uint32_t)__popc(units) * 4096u);
            }
            __syncwarp();
            if (valid) {
                const uint32_t dst = sbase + (uint32_t)s * SB_TILE + (uint32_t)(lane & 7) * 2048u;
                tma_load_3d(dst, &kmap, 0, sl, (int)pp, bar + 8u * s);
                tma_load_3d(dst + SB_HALF, &kmap, 64, sl, (int)pp, bar + 8u * s);
            }
            issued = jl + 1;
        }
        // on a normal exit every stage issued was consumed; after a timeout, let the copies land
        for (int64_t j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
            mbar_wait(bar + 8u * (uint32_t)(j % S), (uint32_t)((j / S) & 1));
    } else if (warp == 1) {
        // ---------------------------------------------------------------- query + MMA
        const uint32_t idesc = idesc_bf16_f32(SB_ROWS, a.N, false);
        const uint32_t qaddr = sbase + L.q;
        const uint32_t qhalf = (uint32_t)a.N * 128u;
        TileCursor c;
        int qr = -1;
        uint32_t qph = 0;
        bool ok = true;
        for (int64_t jl = 0; jl < nk && ok; ++jl) {
            if (!c.seek(a, m0 + jl)) break;
            if (c.r != qr) {
                if (qr >= 0) {  // the MMAs that read the previous query have completed
                    if (lane == 0) tc_commit(qbar);
                    __syncwarp();
                    ok = mbar_wait(qbar, qph);
                    qph ^= 1;
                    if (!ok) break;
                }
                // B row p * HI + h = head h of position p (zero for h >= Hi and past the
                // positions), K-major with 128-byte swizzle: chunk cc of half kh at
                // half + row * 128 + ((cc ^ (row & 7)) << 4)
                for (int i = lane; i < a.N * 16; i += 32) {
                    const int n = i >> 4, ch = i & 15, p = n / HI, h = n % HI;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (p < a.nq && h < a.Hi)
                        v = __ldg(reinterpret_cast<const uint4*>(
                                      a.q_idx + (((int64_t)c.r * a.nq + p) * a.Hi + h) * DI) + ch);
                    st_shared_v4(qaddr + (uint32_t)(ch >> 3) * qhalf + (uint32_t)n * 128u +
                                     ((uint32_t)((ch & 7) ^ (n & 7)) << 4),
                                 v);
                }
                fence_proxy_async_smem();
                __syncwarp();
                qr = c.r;
            }
            const int s = (int)(jl % S);
            const int buf = (int)(jl & 1);
            if (jl >= 2 && !mbar_wait(accempty + 8u * buf, (uint32_t)(((jl >> 1) & 1) ^ 1))) ok = false;
            if (ok && !mbar_wait(bar + 8u * s, (uint32_t)((jl / S) & 1))) ok = false;
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
                const uint32_t d = tmem + (uint32_t)buf * NT;
                const uint32_t st = sbase + (uint32_t)s * SB_TILE;
#pragma unroll
                for (int kh = 0; kh < 2; ++kh)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint64_t ad = sdesc_sw128(st + (uint32_t)kh * SB_HALF + ks * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(qaddr + (uint32_t)kh * qhalf + ks * 32, 16, 1024);
                        tc_mma_f16(d, ad, bd, idesc, (kh | ks) ? 1u : 0u);
                    }
                tc_commit(bar + 48u + 8u * s);
                tc_commit(accfull + 8u * buf);
            }
            __syncwarp();
        }
        if (!ok) raise_status(a.status, CSA_ERR_TIMEOUT);
        if (qr >= 0) {  // every MMA has completed before the tensor memory is freed
            if (lane == 0) tc_commit(qbar);
            __syncwarp();
            mbar_wait(qbar, qph);
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        const int qw = warp & 3;          // TMEM lane quarter
        const int grp = (warp - 2) >> 2;  // tiles with accumulator buffer grp (jl & 1 == grp)
        const int row = qw * 32 + lane;   // the candidate of the tile this thread takes
        float* wv = reinterpret_cast<float*>(sm + L.cst + (warp - 2) * 512);  // [SB_NQ * HI] weights
        float* cv = wv + SB_NQ * 16;                                  // [SB_NQ] bound factors
        int64_t* gv = reinterpret_cast<int64_t*>(cv + SB_NQ);          // [SB_NQ] candidates
        uint32_t eph = 0;
        bool ok = true, waited = false;
        // all epilogue warps meet (an mbarrier: the wait is bounded)
        auto rendezvous = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(ebar);
            const bool r = mbar_wait(ebar, eph);
            eph ^= 1;
            return r;
        };
        auto flush = [&](int r) {  // request r's histograms into the global ones, 4 bins at a time
            if (!waited) {  // the global histograms are cleared by the preceding kernel of the step
                pdl_wait();
                waited = true;
            }
            // one bulk reduction per position by the copy engine (the counts were made visible to
            // it by every epilogue thread's proxy fence before the rendezvous)
            if (threadIdx.x == 64) {
                for (int p = 0; p < a.nq; ++p)
                    bulk_red_add_u32(a.hist + ((int64_t)r * a.nq + p) * kHistBlock,
                                     smem_u32(hist) + 4u * (uint32_t)(p << a.hb), 4u << a.hb);
                bulk_commit();
                bulk_wait_read_all();
            }
        };
        auto zero_hist = [&]() {  // after a rendezvous that follows the flush
            for (int i = (int)threadIdx.x - 64; i < (a.nq << a.hb) / 4; i += SB_FLUSH_T)
                st_shared_zero16(smem_u32(hist) + 16u * (uint32_t)i);
        };
        TileCursor c;
        int er = -1;
        for (int64_t jl = 0; jl < nk; ++jl) {
            if (!c.seek(a, m0 + jl)) break;
            if (c.r != er) {
                if (er >= 0 && a.hist) {
                    fence_proxy_async_smem();
                    ok = rendezvous();
                    if (ok) flush(er);
                    ok = ok && rendezvous();
                    if (ok) zero_hist();
                    ok = ok && rendezvous();
                    if (!ok) break;
                }
                // request c.r's weights (column layout) and, per position, the bound's factor
                for (int i = lane; i < SB_NQ * HI; i += 32) {
                    const int p = i / HI, h = i % HI;
                    wv[i] = (p < a.nq && h < a.Hi) ? __ldg(a.w_h + ((int64_t)c.r * a.nq + p) * a.Hi + h) : 0.f;
                }
                for (int p = 0; p < a.nq; ++p) {
                    float part = 0.f;
                    if (lane < a.Hi) {
                        const int64_t e = (int64_t)c.r * a.nq + p;
                        const uint4* src = reinterpret_cast<const uint4*>(a.q_idx + (e * a.Hi + lane) * DI);
                        float l1 = 0.f;
#pragma unroll 4
                        for (int i = 0; i < 16; ++i) l1 += abs_sum8(__ldg(src + i));
                        part = fabsf(__ldg(a.w_h + e * a.Hi + lane)) * l1;
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                    if (lane == 0) {
                        cv[p] = part * (SB_MARGIN * 1.001f);  // the factor covers these sums' rounding
                        gv[p] = a.n_tokens ? query_tokens(a.n_tokens, c.r * a.nq + p, a.nq) / a.ratio : a.G;
                    }
                }
                __syncwarp();
                er = c.r;
            }
            const int buf = (int)(jl & 1);
            if (buf != grp) continue;  // the other group's tile
            const int s = (int)(jl % S);
            if (!mbar_wait(bar + 8u * s, (uint32_t)((jl / S) & 1)) ||
                !mbar_wait(accfull + 8u * buf, (uint32_t)((jl >> 1) & 1))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t d[NT];
#pragma unroll
            for (int c16 = 0; c16 < NT / 16; ++c16)
                tc_ld16(tmem + ((uint32_t)(qw * 32) << 16) + (uint32_t)buf * NT + c16 * 16, d + 16 * c16);
            tc_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(accempty + 8u * buf);
            // max |k| over the candidate's row: its 16 chunks in any order -- physical chunk
            // ch ^ (row & 7) at step ch, so that the 8 rows of a load phase hit 8 bank groups
            const uint32_t rb = sbase + (uint32_t)s * SB_TILE + (uint32_t)row * 128u;
            uint32_t mx = 0;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 v = ld_shared_v4(rb + (uint32_t)h2 * SB_HALF + (uint32_t)((ch ^ row) & 7) * 16u);
                    mx = __vmaxu2(mx, v.x & 0x7FFF7FFFu);
                    mx = __vmaxu2(mx, v.y & 0x7FFF7FFFu);
                    mx = __vmaxu2(mx, v.z & 0x7FFF7FFFu);
                    mx = __vmaxu2(mx, v.w & 0x7FFF7FFFu);
                }
            const uint32_t mk = (mx & 0xFFFFu) > (mx >> 16) ? (mx & 0xFFFFu) : (mx >> 16);
            const bool page_ok = (umask[s] >> (row >> 4)) & 1u;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar + 48u + 8u * s);
            const float M = __uint_as_float(mk << 16);
            const int64_t g = (m0 + jl - c.base) * SB_ROWS + row;
#pragma unroll
            for (int p = 0; p < SB_NQ; ++p) {
                if (p >= a.nq) break;
                const bool in = g < gv[p];
                float up = 0.f, lo = 0.f;
                if (page_ok) {
                    bool bad = mk >= 0x7F80u;
                    float sh = 0.f;
#pragma unroll
                    for (int h = 0; h < HI; ++h) {
                        const float x = __uint_as_float(d[p * HI + h]);
                        bad |= !(fabsf(x) <= FLT_MAX);
                        sh = __fmaf_rn(wv[p * HI + h], x > 0.f ? x : 0.f, sh);
                    }
                    const float e = __fmaf_ru(cv[p], M, 1e-30f);
                    bad |= !(e <= 1e30f) || !(fabsf(sh) <= FLT_MAX);
                    up = bad ? INFINITY : __fadd_ru(sh, e);
                    lo = bad ? -INFINITY : __fsub_rd(sh, e);
                }
                const int64_t o = ((int64_t)c.r * a.nq + p) * a.score_stride + g;
                if (in) {
                    a.upper[o] = up;
                    if (a.lower) a.lower[o] = lo;
                }
                // 4K-16K bins over scattered scores: the lanes' bins rarely coincide, so plain
                // shared-memory atomics (no warp aggregation)
                if (a.hist && in) atomicAdd(&hist[(p << a.hb) + (score_key(lo) >> (32 - a.hb))], 1u);
            }
        }
        if (!ok) raise_status(a.status, CSA_ERR_TIMEOUT);
        if (ok && er >= 0 && a.hist) {
            fence_proxy_async_smem();
            if (rendezvous()) flush(er);
            else raise_status(a.status, CSA_ERR_TIMEOUT);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TCOLS);
}

// ------------------------------------------------------------------ host side
bool score_bound_supported(int Hi, int nq, bool fp8) { return !fp8 && Hi >= 1 && Hi <= 16 && nq >= 1 && nq <= SB_NQ; }

template <int HI>
static cudaError_t launch_bound_t(const CUtensorMap& map, BoundArgs a, int64_t tiles_bound, cudaStream_t s,
                                  bool pdl) {
    constexpr uint32_t kMaxSmem = 225 * 1024;  // leaves room for the static shared memory
    int S = SB_MAX_STAGES;
    BoundLayout L = bound_layout(S, a.N, a.nq, a.hist != nullptr, a.hb);
    while (L.total > kMaxSmem && S > 2) L = bound_layout(--S, a.N, a.nq, a.hist != nullptr, a.hb);
    if (L.total > kMaxSmem) return cudaErrorInvalidValue;
    a.S = S;
    // one value for every configuration: the attribute is the kernel's, not the launch's
    cudaError_t e = set_func_attr_once((const void*)score_bound_kernel<HI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    int64_t grid = sms;
    if (tiles_bound < grid) grid = tiles_bound < 1 ? 1 : tiles_bound;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(SB_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, score_bound_kernel<HI>, map, a);
}

cudaError_t launch_score_bound(const ScoreLaunch& h, float* lower, cudaStream_t s, bool pdl) {
    const int nq = h.nq > 1 ? h.nq : 1;
    if (!score_bound_supported(h.Hi, nq, h.fp8)) return cudaErrorInvalidValue;
    const int hi = h.Hi <= 4 ? 4 : (h.Hi <= 8 ? 8 : 16);
    BoundArgs a;
    a.q_idx = static_cast<const uint16_t*>(h.q_idx);
    a.w_h = h.w_h;
    a.Hi = h.Hi;
    a.nq = nq;
    a.N = (nq * hi + 15) / 16 * 16;
    a.pt = h.kidx.pt;
    a.pt_stride = h.kidx.pt_stride;
    a.upper = h.scores;
    a.lower = lower;
    a.score_stride = h.score_stride;
    a.B = h.n_tokens ? h.B / nq : 1;  // requests (the launch's B counts batch entries)
    a.n_tokens = h.n_tokens;
    a.ratio = h.ratio;
    a.G = h.G;
    a.hist = h.hist;
    a.hb = bound_hist_bits(nq);
    a.status = h.status;
    a.S = SB_MAX_STAGES;
    int64_t rpp, n_pages;
    if (h.kidx.pt) {
        rpp = h.kidx.rpp;
        n_pages = h.kidx.n_pages;
    } else {  // contiguous rows: a single "page" holding every row
        rpp = h.max_G > 0 ? h.max_G : 1;
        n_pages = 1;
    }
    a.rpp = (int32_t)rpp;
    a.n_pages = n_pages;
    CUtensorMap map;
    if (!make_kidx_map(&map, h.kidx, false, rpp, n_pages)) return cudaErrorInvalidValue;
    const int64_t tiles = (int64_t)a.B * ((h.max_G + SB_ROWS - 1) / SB_ROWS);
    if (hi == 4) return launch_bound_t<4>(map, a, tiles, s, pdl);
    if (hi == 8) return launch_bound_t<8>(map, a, tiles, s, pdl);
    return launch_bound_t<16>(map, a, tiles, s, pdl);
}

}  // namespace csa
