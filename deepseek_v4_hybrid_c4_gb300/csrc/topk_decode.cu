// Stage 3 of the decode step: the exact top-k set of every request's index scores ("SGLang
// 如何为 DeepSeek V4 打造「Day-0」推理加速", sec. "创新 2", Lightning TopK: histograms give a
// threshold bin, then a scatter of the entries above it), laid out for a one-token decode
// step where the whole select sits on the critical path between the score kernel and the
// attention.
//
// Order, as in the cluster select: descending order-preserving key of the fp32 score, ties
// to the lower index -- descending composite V = key << 31 | (2^31 - 1 - index), digits
// key 31..21 | 20..10 | 9..0, then inverted index 30..20 | 19..10 | 9..0.
//
// A wide grid instead of one cluster: request b gets C CTAs of SW_T threads, CTA c owning
// the SW_SLICE scores [c SW_SLICE, (c+1) SW_SLICE), four per thread (one 16-byte load), so
// the 1 MB of scores of a 262,144-candidate request is read by 128 SMs at once.  Two
// kernels, chained by programmatic dependent launch:
//  scan:   every CTA reads the first digit's histogram, which the score kernel built, and
//          finds the bin b0 holding the k-th key.  Its keys above b0 are winners, keys in b0
//          candidates; both lists go, in index order, to the CTA's own region of the
//          workspace (winners first), the candidates' second digit is counted into a global
//          histogram, and the CTA publishes its two counts.
//  finish: every CTA takes the prefix sums of the published counts and writes its own
//          region's winners.  Every CTA also finds the second digit's bin b1 in the global
//          histogram.  When taking all of b1 completes the set (the usual case), every CTA
//          counts each region's candidates with a second digit >= b1, warp by warp with
//          ballots, and writes its own region's at the prefix of those counts -- no CTA waits
//          for another.  Otherwise CTA 0 loads all candidates (index order; into shared memory
//          when they fit) and refines them digit by digit -- the others counted in shared
//          memory -- appending each round's winners in index order until the threshold bin
//          holds exactly the number still needed.
// Output: the k indices as a set in a fixed order (first-digit winners, then each round's
// winners, each in index order); -1 pads when the request has fewer than k candidates.
#include <cstddef>

#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int SW_T = 512;                 // threads per CTA
constexpr int SW_PER = 4;                 // scores per thread
constexpr int SW_SLICE = SW_T * SW_PER;   // scores per CTA
constexpr int SW_CAP = 8192;              // candidates the last CTA keeps in shared memory
constexpr int SW_CMAX = 2048;             // CTAs per request
constexpr int SW_BINS = kHistBins;        // 2048: widest digit
// Shared memory the scan kernel reserves without using it: more than half an SM's, so the
// scan CTAs spread one per SM (each then has an SM's load slots for its 2,048 scores) and
// still leave room for a finish CTA waiting on the same SM.
constexpr size_t SW_SCAN_SPREAD_SMEM = 116 * 1024;

struct SelArgs {
    int nq;  // decode mode: query positions per request (batch entry b: request b / nq)
    // request b's scores: decode mode (n_tokens): scores + b * score_stride, n_tokens[b] / ratio
    // of them; offsets mode: [offsets[b], offsets[b+1]); single: [0, G)
    const float* scores;
    int64_t score_stride;
    const int64_t* n_tokens;
    int ratio;
    const int64_t* offsets;
    int64_t G;
    int sorted;              // 1: output ordered by (score desc, index asc) (standalone calls)
    uint32_t* keys_out;      // [B][k] or nullptr (sorted output only)
    int C;                   // CTAs per request
    int k;
    int32_t* out;            // [B][k]
    uint32_t* hist;          // [B][kHistBlock]: digit 0 from the score kernel; digit 1 and the counter here
    uint64_t* lists;         // [B][C * SW_SLICE]: per CTA, winners then candidates, key << 32 | index
                             // (after the tensor-core bounds: [B][C * SB_SLICE], see slice)
    int slice = 0;           // region stride of lists for the exact select (SB_SLICE)
    uint32_t* counts;        // [B][C]: winners << 16 | candidates
    int32_t* status;
};

struct SwCore {              // scans and bin searches
    uint32_t wsum[SW_T / 32];
    uint64_t wsum64[SW_T / 32];
    uint32_t bin, above, cnt;
};

struct SwFinSmem {           // finish kernel
    SwCore core;
    uint32_t wpre[SW_CMAX + 1];  // exclusive prefix of the CTAs' winners (wpre[C] = total)
    uint32_t cpre[SW_CMAX + 1];  // ... and of their candidates
    uint32_t spre[SW_CMAX + 1];  // per region: candidates taken in the second digit, then their prefix
    uint32_t hist[SW_BINS];
    uint2 cand[SW_CAP];      // candidates (slow path, CTA 0): {key, index}; sorted output: the
                             // selected composites (first 2048 slots) and this CTA's own (next 2048)
    uint32_t ntk, nown;
};

// 63-bit composite of a list entry key << 32 | index: larger = earlier in the output.
__device__ __forceinline__ uint64_t sel_comp(uint64_t v) {
    return (v & 0xFFFFFFFF00000000ull) | (0x7FFFFFFFu - (uint32_t)v);
}

__device__ __forceinline__ void sel_span(const SelArgs& a, int b, const float*& sc, int64_t& G) {
    if (a.n_tokens) {
        sc = a.scores + (int64_t)b * a.score_stride;
        G = query_tokens(a.n_tokens, b, a.nq) / a.ratio;
    } else if (a.offsets) {
        const int64_t o0 = __ldg(a.offsets + b), o1 = __ldg(a.offsets + b + 1);
        sc = a.scores + o0;
        G = o1 - o0;
    } else {
        sc = a.scores;
        G = a.G;
    }
    if (G < 0) G = 0;
}

// Keys of the four scores pos .. pos + 3 (one 16-byte load when aligned and in range); key 0
// past the end.
__device__ __forceinline__ void sel_load4(const float* sc, int64_t pos, int64_t G, uint32_t (&key)[SW_PER]) {
    if (pos + SW_PER - 1 < G && (reinterpret_cast<uintptr_t>(sc + pos) & 15) == 0) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(sc + pos));
        key[0] = score_key(f.x);
        key[1] = score_key(f.y);
        key[2] = score_key(f.z);
        key[3] = score_key(f.w);
    } else {
#pragma unroll
        for (int q = 0; q < SW_PER; ++q) key[q] = pos + q < G ? score_key(__ldcg(sc + pos + q)) : 0u;
    }
}

// Exclusive prefix of v over the CTA's threads; *total = the sum.  Every thread calls it.
__device__ __forceinline__ uint32_t sw_scan(SwCore& sm, uint32_t v, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.wsum[warp] = x;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SW_T / 32; ++w) {
        const uint32_t s = sm.wsum[w];
        before += w < warp ? s : 0u;
        tot += s;
    }
    __syncthreads();  // wsum is free again
    *total = tot;
    return before + x - v;
}

// The same over 64-bit values.
__device__ __forceinline__ uint64_t sw_scan64(SwCore& sm, uint64_t v, uint64_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.wsum64[warp] = x;
    __syncthreads();
    uint64_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < SW_T / 32; ++w) {
        const uint64_t s = sm.wsum64[w];
        before += w < warp ? s : 0ull;
        tot += s;
    }
    __syncthreads();
    *total = tot;
    return before + x - v;
}

// The bin holding the need-th largest element, counting from the top bin, given thread t's
// four bins 2047 - 4t - j (j = 0..3, high first).  Sets sm.bin (~0 when the counts hold
// fewer than need), sm.above (elements in higher bins) and sm.cnt (elements in the bin).
__device__ __forceinline__ void sw_find_bin(SwCore& sm, const uint32_t (&h)[4], uint32_t need) {
    if (threadIdx.x == 0) {
        sm.bin = ~0u;
        sm.above = 0;
        sm.cnt = 0;
    }
    uint32_t tot;
    uint32_t acc = sw_scan(sm, h[0] + h[1] + h[2] + h[3], &tot);  // its barriers order the reset
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (h[j] > 0 && acc < need && need <= acc + h[j]) {
            sm.bin = (uint32_t)(SW_BINS - 1 - 4 * (int)threadIdx.x - j);
            sm.above = acc;
            sm.cnt = h[j];
        }
        acc += h[j];
    }
    __syncthreads();
}

// Digit d (1..5) of the composite of (key, index).
__device__ __forceinline__ uint32_t sw_digit(int d, uint32_t key, int32_t idx) {
    const uint32_t inv = 0x7FFFFFFFu - (uint32_t)idx;
    switch (d) {
        case 1: return (key >> 10) & 2047u;
        case 2: return key & 1023u;
        case 3: return (inv >> 20) & 2047u;
        case 4: return (inv >> 10) & 1023u;
        default: return inv & 1023u;
    }
}

// Largest c in [0, C) with pre[c] <= x (pre non-decreasing, pre[0] = 0).
__device__ __forceinline__ int sw_owner(const uint32_t* pre, int C, uint32_t x) {
    int lo = 0, n = C;
    while (n > 1) {
        const int h = n >> 1;
        if (pre[lo + h] <= x) lo += h;
        n -= h;
    }
    return lo;
}

__global__ void __launch_bounds__(SW_T) select_scan_kernel(SelArgs a) {
    __shared__ SwCore sm;
    const int tid = threadIdx.x;
    const int b = blockIdx.x, c = blockIdx.y, C = a.C, k = a.k;
    const float* sc;
    int64_t G;
    sel_span(a, b, sc, G);
    uint32_t* hb = a.hist + (int64_t)b * kHistBlock;
    uint64_t* lc = a.lists + ((int64_t)b * C + c) * SW_SLICE;
    const bool all_in = G <= k;
    pdl_wait();  // the scores and the first digit's histogram come from the score kernel
    pdl_launch_dependents();
    if ((int64_t)c * SW_SLICE >= G && c > 0) {  // a slice past a shorter request's end: nothing in it
        if (tid == 0) a.counts[(int64_t)b * C + c] = 0u;
        return;
    }

    // ---- this thread's four keys, and the first digit's bin
    const int64_t pos = (int64_t)c * SW_SLICE + SW_PER * tid;
    uint32_t key[SW_PER];
    sel_load4(sc, pos, G, key);
    uint32_t b0 = 0;
    if (!all_in) {
        const uint4 hv = __ldcg(reinterpret_cast<const uint4*>(hb + (SW_BINS - 4 - 4 * tid)));
        const uint32_t h[4] = {hv.w, hv.z, hv.y, hv.x};
        sw_find_bin(sm, h, (uint32_t)k);
        b0 = sm.bin;  // ~0u (inconsistent histogram): no winners, no candidates; the finish reports it
    }

    // ---- winners and candidates of the slice, in index order, to this CTA's region
    bool win[SW_PER], cand[SW_PER];
    uint32_t nw = 0, nc = 0;
#pragma unroll
    for (int q = 0; q < SW_PER; ++q) {
        const bool in = pos + q < G;
        const uint32_t d0 = key[q] >> 21;
        win[q] = in && (all_in || d0 > b0);
        cand[q] = in && !all_in && d0 == b0;
        nw += win[q] ? 1u : 0u;
        nc += cand[q] ? 1u : 0u;
    }
    uint32_t tot;
    const uint32_t ex = sw_scan(sm, (nw << 16) | nc, &tot);
    const uint32_t tw = tot >> 16, tc = tot & 0xFFFFu;
    uint32_t ow = ex >> 16, oc = tw + (ex & 0xFFFFu);
#pragma unroll
    for (int q = 0; q < SW_PER; ++q) {
        const uint64_t v = ((uint64_t)key[q] << 32) | (uint32_t)(pos + q);
        if (win[q]) {
            lc[ow++] = v;
        } else if (cand[q]) {
            lc[oc++] = v;
            atomicAdd(hb + SW_BINS + ((key[q] >> 10) & 2047u), 1u);
        }
    }
    if (tid == 0) a.counts[(int64_t)b * C + c] = (tw << 16) | tc;
}

// At most 88 registers: 512 x 88 plus a scan CTA's 512 x 40 fill the register file exactly, so a
// finish CTA becomes resident beside its SM's scan CTA and waits there (no spills at this cap).
// A grid of more CTAs than SMs but at most twice as many takes the 64-register instance instead
// (two finish CTAs per SM, one wave; it spills a little): speculative verify with two query
// positions, 70.8 -> 68.8 us.  Larger grids (the 32-request ragged batch) keep 88.
template <int MAXREG>
__global__ void __maxnreg__(MAXREG) select_finish_kernel(SelArgs a) {
    extern __shared__ __align__(16) uint8_t sw_raw[];
    SwFinSmem& fs = *reinterpret_cast<SwFinSmem*>(sw_raw);
    SwCore& sm = fs.core;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = SW_T / 32;
    const int b = blockIdx.x, c = blockIdx.y, C = a.C, k = a.k;
    const float* sc_unused;
    int64_t G;
    sel_span(a, b, sc_unused, G);
    const uint32_t* hb = a.hist + (int64_t)b * kHistBlock;
    const uint64_t* lb = a.lists + (int64_t)b * C * SW_SLICE;
    const uint32_t* cb = a.counts + (int64_t)b * C;
    int32_t* out = a.out + (int64_t)b * k;
    const bool all_in = G <= k;
    pdl_wait();  // the lists, their counts and the second digit's histogram come from the scan
    pdl_launch_dependents();
    if ((int64_t)c * SW_SLICE >= G && c > 0) return;  // an empty region (a shorter request): nothing to place
    // entry tid of this CTA's own region, read with the counts: it holds the region's winners
    // and candidates whenever they number at most SW_T (the other entries go unused)
    const uint64_t* lc = lb + (int64_t)c * SW_SLICE;
    const uint64_t mine = __ldcg(lc + tid);

    // ---- offsets of every CTA's lists: thread t owns CTAs [t g, t g + g)
    const int g = (C + SW_T - 1) / SW_T;  // <= 4
    uint32_t cw[4], cn[4], sw_ = 0, sc_ = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int cj = tid * g + j;
        const uint32_t v = (j < g && cj < C) ? __ldcg(cb + cj) : 0u;
        cw[j] = v >> 16;
        cn[j] = v & 0xFFFFu;
        sw_ += cw[j];
        sc_ += cn[j];
    }
    uint32_t h1[4] = {0u, 0u, 0u, 0u};  // the candidates' second digit, counted by every scan CTA
    if (!all_in) {
        const uint4 hv = __ldcg(reinterpret_cast<const uint4*>(hb + SW_BINS + (SW_BINS - 4 - 4 * tid)));
        h1[0] = hv.w;
        h1[1] = hv.z;
        h1[2] = hv.y;
        h1[3] = hv.x;
    }
    uint64_t tot64;
    const uint64_t x64 = sw_scan64(sm, ((uint64_t)sw_ << 32) | sc_, &tot64);  // winners high, candidates low
    const uint32_t W0 = (uint32_t)(tot64 >> 32), Cn = (uint32_t)tot64;
    uint32_t xw = (uint32_t)(x64 >> 32), xc = (uint32_t)x64;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int cj = tid * g + j;
        if (j < g && cj < C) {
            fs.wpre[cj] = xw;
            fs.cpre[cj] = xc;
            xw += cw[j];
            xc += cn[j];
        }
    }
    if (tid == 0) {
        fs.wpre[C] = W0;
        fs.cpre[C] = Cn;
    }
    __syncthreads();
    const bool ok = all_in ? W0 == (uint32_t)G : (W0 < (uint32_t)k && W0 + Cn >= (uint32_t)k);
    if (!ok) {  // the histogram does not match the scores (not cleared, or written by another step)
        if (c == 0) {
            if (tid == 0) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
            for (int i = tid; i < k; i += SW_T) out[i] = -1;
        }
        return;
    }
    // ---- this CTA's first-digit winners
    const uint32_t my_w = fs.wpre[c + 1] - fs.wpre[c], my_c = fs.cpre[c + 1] - fs.cpre[c];
    const bool sorted = a.sorted != 0;
    uint64_t* tk = reinterpret_cast<uint64_t*>(fs.cand);  // sorted output: every selected composite
    uint64_t* own = tk + 2048;                            // ... and this CTA's
    if (!sorted) {
        if ((uint32_t)tid < my_w) out[fs.wpre[c] + tid] = (int32_t)(uint32_t)mine;
        for (uint32_t i = SW_T + tid; i < my_w; i += SW_T) out[fs.wpre[c] + i] = (int32_t)(uint32_t)__ldcg(lc + i);
    }
    if (tid == 0) {
        fs.ntk = 0;
        fs.nown = 0;
    }
    __syncthreads();
    // Sorted output: with every selected composite in tk[0, ntk) and this CTA's own in
    // own[0, nown), a warp per own entry counts the larger ones -- its output position.
    auto rank_own = [&]() {
        __syncthreads();
        const uint32_t ntk = fs.ntk, nown = fs.nown;
        for (uint32_t e = warp; e < nown; e += NW) {
            const uint64_t x = own[e];
            uint32_t r = 0;
            for (uint32_t j = lane; j < ntk; j += 32) r += tk[j] > x ? 1u : 0u;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
            if (lane == 0 && r < (uint32_t)k) {
                out[r] = (int32_t)(0x7FFFFFFFu - (uint32_t)x);
                if (a.keys_out) a.keys_out[(int64_t)b * k + r] = (uint32_t)(x >> 32);
            }
        }
    };
    if (all_in) {
        if (sorted) {  // every score is selected: gather every region's (winners-only) list
            for (int cb0 = warp; cb0 < C; cb0 += 8 * NW) {
                uint32_t n8[8], nmax = 0;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int cj = cb0 + u * NW;
                    n8[u] = cj < C ? fs.wpre[cj + 1] - fs.wpre[cj] : 0u;
                    nmax = max(nmax, n8[u]);
                }
                for (uint32_t i0 = 0; i0 < nmax; i0 += 32) {
                    const uint32_t i = i0 + lane;
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (i < n8[u])
                            tk[atomicAdd(&fs.ntk, 1u)] = sel_comp(__ldcg(lb + (int64_t)(cb0 + u * NW) * SW_SLICE + i));
                }
            }
            for (uint32_t i = tid; i < my_w; i += SW_T)
                own[atomicAdd(&fs.nown, 1u)] = sel_comp(i < (uint32_t)SW_T ? mine : __ldcg(lc + i));
            rank_own();
        }
        if (c == 0)
            for (int i = (int)W0 + tid; i < k; i += SW_T) {
                out[i] = -1;
                if (sorted && a.keys_out) a.keys_out[(int64_t)b * k + i] = 0u;
            }
        return;
    }
    uint32_t need = (uint32_t)k - W0, base = W0;
    sw_find_bin(sm, h1, need);
    const uint32_t bd1 = sm.bin, above1 = sm.above, cnt1 = sm.cnt;
    if (bd1 == ~0u) {  // cannot happen: the candidates hold at least `need` elements
        if (c == 0) {
            if (tid == 0) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
            for (int i = (int)base + tid; i < k; i += SW_T) out[i] = -1;
        }
        return;
    }

    if (cnt1 == need - above1) {
        // ---- fast path: the candidates whose second digit is >= bd1 complete the set.  Count
        //      them per region (warp w: regions w, w + 16, ..., eight in flight per lane) ...
        //      (sorted output: whole regions, winners included, and every selected composite
        //      goes to tk)
        for (int cb0 = warp; cb0 < C; cb0 += 8 * NW) {
            uint32_t nw8[8], off8[8], n8[8], t8[8], nmax = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cj = cb0 + u * NW;
                nw8[u] = cj < C ? fs.wpre[cj + 1] - fs.wpre[cj] : 0u;
                off8[u] = sorted ? 0u : nw8[u];
                n8[u] = (cj < C ? fs.cpre[cj + 1] - fs.cpre[cj] : 0u) + (sorted ? nw8[u] : 0u);
                t8[u] = 0u;
                nmax = max(nmax, n8[u]);
            }
            for (uint32_t i0 = 0; i0 < nmax; i0 += 32) {
                const uint32_t i = i0 + lane;
                uint64_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i < n8[u]) v[u] = __ldcg(lb + (int64_t)(cb0 + u * NW) * SW_SLICE + off8[u] + i);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const bool is_cand = off8[u] + i >= nw8[u];
                    const bool t = i < n8[u] && is_cand && ((uint32_t)(v[u] >> 42) & 2047u) >= bd1;
                    t8[u] += (uint32_t)__popc(__ballot_sync(0xffffffffu, t));
                    if (sorted && i < n8[u] && (t || !is_cand)) tk[atomicAdd(&fs.ntk, 1u)] = sel_comp(v[u]);
                }
            }
            if (lane == 0)
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (cb0 + u * NW < C) fs.spre[cb0 + u * NW] = t8[u];
        }
        __syncthreads();
        // ... their prefix over the regions ...
        uint32_t st[4], ss = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cj = tid * g + j;
            st[j] = (j < g && cj < C) ? fs.spre[cj] : 0u;
            ss += st[j];
        }
        uint32_t taken;
        uint32_t xs = sw_scan(sm, ss, &taken);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cj = tid * g + j;
            if (j < g && cj < C) {
                fs.spre[cj] = xs;
                xs += st[j];
            }
        }
        __syncthreads();
        if (c == 0 && tid == 0 && taken != need) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
        if (sorted) {  // this CTA's selected entries, ranked among all of them
            for (uint32_t i = tid; i < my_w + my_c; i += SW_T) {
                const uint64_t v = i < (uint32_t)SW_T ? mine : __ldcg(lc + i);
                if (i < my_w || ((uint32_t)(v >> 42) & 2047u) >= bd1) own[atomicAdd(&fs.nown, 1u)] = sel_comp(v);
            }
            if (c == 0 && tid == 0 && fs.ntk != (uint32_t)k) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
            rank_own();
            return;
        }
        // ... and this CTA's own, in index order after every earlier region's
        const uint32_t o0 = base + fs.spre[c];
        if (my_w + my_c <= (uint32_t)SW_T) {  // they sit in `mine` of threads my_w .. my_w + my_c - 1
            const bool t = (uint32_t)tid >= my_w && (uint32_t)tid < my_w + my_c &&
                           ((uint32_t)(mine >> 42) & 2047u) >= bd1;
            uint32_t tt;
            const uint32_t r = o0 + sw_scan(sm, t ? 1u : 0u, &tt);
            if (t && r < (uint32_t)k) out[r] = (int32_t)(uint32_t)mine;
        } else if (warp == 0) {
            uint32_t o = o0;
            for (uint32_t i0 = 0; i0 < my_c; i0 += 32) {
                const uint32_t i = i0 + lane;
                const uint64_t v = i < my_c ? __ldcg(lc + my_w + i) : 0ull;
                const bool t = i < my_c && ((uint32_t)(v >> 42) & 2047u) >= bd1;
                const unsigned m = __ballot_sync(0xffffffffu, t);
                const uint32_t r = o + (uint32_t)__popc(m & ((1u << lane) - 1u));
                if (t && r < (uint32_t)k) out[r] = (int32_t)(uint32_t)v;
                o += (uint32_t)__popc(m);
            }
        }
        return;
    }

    // ---- general path (ties at the threshold, wide bins): CTA 0 refines every candidate
    if (c != 0) return;
    if (sorted) {  // the first-digit winners were not written: every region's, in fixed order
        for (int r = warp; r < C; r += NW) {
            const uint32_t n = fs.wpre[r + 1] - fs.wpre[r];
            for (uint32_t i = lane; i < n; i += 32)
                out[fs.wpre[r] + i] = (int32_t)(uint32_t)__ldcg(lb + (int64_t)r * SW_SLICE + i);
        }
    }
    const bool held = Cn <= (uint32_t)SW_CAP;
    auto cand_src = [&](uint32_t j) {
        const int cj = sw_owner(fs.cpre, C, j);
        return lb + (int64_t)cj * SW_SLICE + (fs.wpre[cj + 1] - fs.wpre[cj]) + (j - fs.cpre[cj]);
    };
    if (held) {  // every region at once: warp w copies regions w, w + 16, ... (eight in flight per lane)
        for (int cb0 = warp; cb0 < C; cb0 += 8 * NW) {
            uint32_t off8[8], co8[8], n8[8], nmax = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int cj = cb0 + u * NW;
                off8[u] = cj < C ? fs.wpre[cj + 1] - fs.wpre[cj] : 0u;
                co8[u] = cj < C ? fs.cpre[cj] : 0u;
                n8[u] = cj < C ? fs.cpre[cj + 1] - co8[u] : 0u;
                nmax = max(nmax, n8[u]);
            }
            for (uint32_t i0 = 0; i0 < nmax; i0 += 32) {
                const uint32_t i = i0 + lane;
                uint64_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i < n8[u]) v[u] = __ldcg(lb + (int64_t)(cb0 + u * NW) * SW_SLICE + off8[u] + i);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    if (i < n8[u]) fs.cand[co8[u] + i] = make_uint2((uint32_t)(v[u] >> 32), (uint32_t)v[u]);
            }
        }
        __syncthreads();
    }
    auto cand_at = [&](uint32_t j, uint32_t& kk, int32_t& ii) {
        if (held) {
            const uint2 e = fs.cand[j];
            kk = e.x;
            ii = (int32_t)e.y;
        } else {
            const uint64_t v = __ldcg(cand_src(j));
            kk = (uint32_t)(v >> 32);
            ii = (int32_t)(uint32_t)v;
        }
    };

    // rounds over digits 1..5 on the candidates (each thread a contiguous range)
    const uint32_t per = (Cn + SW_T - 1) / SW_T;
    const uint32_t j0 = min((uint32_t)tid * per, Cn), j1 = min(j0 + per, Cn);
    uint32_t bins[6] = {0u, 0u, 0u, 0u, 0u, 0u};
    for (int d = 1; d <= 5; ++d) {
        uint32_t bd = bd1, above = above1, cnt = cnt1;
        if (d > 1) {
            uint32_t h[4];
            for (int i = tid; i < SW_BINS; i += SW_T) fs.hist[i] = 0u;
            __syncthreads();
            for (uint32_t j = j0; j < j1; ++j) {
                uint32_t kk;
                int32_t ii;
                cand_at(j, kk, ii);
                bool m = true;
                for (int e = 1; e < d; ++e) m = m && sw_digit(e, kk, ii) == bins[e];
                if (m) atomicAdd(&fs.hist[sw_digit(d, kk, ii)], 1u);
            }
            __syncthreads();
#pragma unroll
            for (int j = 0; j < 4; ++j) h[j] = fs.hist[SW_BINS - 1 - 4 * tid - j];
            sw_find_bin(sm, h, need);
            bd = sm.bin;
            above = sm.above;
            cnt = sm.cnt;
        }
        if (bd == ~0u) {  // cannot happen: the candidates hold at least `need` elements
            if (tid == 0) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
            for (int i = (int)base + tid; i < k; i += SW_T) out[i] = -1;
            return;
        }
        bins[d] = bd;
        const bool last_round = cnt == need - above;  // the whole bin is taken
        if (d == 2 && !last_round) {
            // every key bit is fixed: the bin holds need - above or more candidates of one key,
            // and the tie goes to the lower index -- the first ones in storage order (regions in
            // order, each in index order).  Take them in one pass instead of three index digits.
            const uint32_t need_t = need - above;
            uint32_t na = 0, nt = 0;
            for (uint32_t j = j0; j < j1; ++j) {
                uint32_t kk;
                int32_t ii;
                cand_at(j, kk, ii);
                if (sw_digit(1, kk, ii) != bins[1]) continue;
                const uint32_t dv = sw_digit(2, kk, ii);
                na += dv > bd ? 1u : 0u;
                nt += dv == bd ? 1u : 0u;
            }
            uint32_t tot_t, tot;
            const uint32_t t_before = sw_scan(sm, nt, &tot_t);
            const uint32_t my_t = t_before >= need_t ? 0u : min(nt, need_t - t_before);
            uint32_t o = base + sw_scan(sm, na + my_t, &tot);
            uint32_t taken_t = 0;
            for (uint32_t j = j0; j < j1; ++j) {
                uint32_t kk;
                int32_t ii;
                cand_at(j, kk, ii);
                if (sw_digit(1, kk, ii) != bins[1]) continue;
                const uint32_t dv = sw_digit(2, kk, ii);
                const bool t = dv > bd || (dv == bd && taken_t++ < my_t);
                if (t) {
                    if (o < (uint32_t)k) out[o] = ii;
                    ++o;
                }
            }
            base += tot;
            break;
        }
        // this round's winners in index order: digit above bd (or the whole bin, last round)
        auto takes = [&](uint32_t kk, int32_t ii) {
            for (int e = 1; e < d; ++e)
                if (sw_digit(e, kk, ii) != bins[e]) return false;
            const uint32_t dv = sw_digit(d, kk, ii);
            return dv > bd || (last_round && dv == bd);
        };
        uint32_t n = 0;
        for (uint32_t j = j0; j < j1; ++j) {
            uint32_t kk;
            int32_t ii;
            cand_at(j, kk, ii);
            n += takes(kk, ii) ? 1u : 0u;
        }
        uint32_t rt;
        uint32_t o = base + sw_scan(sm, n, &rt);
        for (uint32_t j = j0; j < j1; ++j) {
            uint32_t kk;
            int32_t ii;
            cand_at(j, kk, ii);
            if (takes(kk, ii)) {
                if (o < (uint32_t)k) out[o] = ii;
                ++o;
            }
        }
        base += rt;
        if (last_round) break;
        need -= above;
    }
    if (base != (uint32_t)k && tid == 0) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    if (!sorted) return;
    // sorted output: order the k entries just written (the candidates are no longer needed, so
    // their space holds the sort), a bitonic sort of the composites, descending
    __syncthreads();
    const float* sc;
    int64_t Gs;
    sel_span(a, b, sc, Gs);
    int n = 1;
    while (n < k) n <<= 1;
    for (int i = tid; i < n; i += SW_T) {
        const int32_t idx = i < k ? out[i] : -1;
        tk[i] = (idx >= 0 && idx < Gs) ? ((uint64_t)score_key(__ldcg(sc + idx)) << 32) | (0x7FFFFFFFu - (uint32_t)idx)
                                       : 0ull;
    }
    __syncthreads();
    for (int size = 2; size <= n; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int p = tid; p < (n >> 1); p += SW_T) {
                const int lo = 2 * p - (p & (stride - 1)), hi = lo + stride;
                const bool desc = (lo & size) == 0;
                const uint64_t x = tk[lo], y = tk[hi];
                if ((x < y) == desc) {
                    tk[lo] = y;
                    tk[hi] = x;
                }
            }
            __syncthreads();
        }
    for (int i = tid; i < k; i += SW_T) {
        const uint64_t x = tk[i];
        out[i] = x ? (int32_t)(0x7FFFFFFFu - (uint32_t)x) : -1;
        if (a.keys_out) a.keys_out[(int64_t)b * k + i] = x ? (uint32_t)(x >> 32) : 0u;
    }
}

// Standalone select, first kernel: clears request blockIdx.x's histogram block (the first
// digit's counts and the candidates' second digit); the histogram kernel loads its scores
// meanwhile and waits for this grid before its first count.
__global__ void __launch_bounds__(256) select_zero_kernel(uint32_t* hist) {
    pdl_launch_dependents();
    uint4* z = reinterpret_cast<uint4*>(hist + (int64_t)blockIdx.x * kHistBlock);
    for (int i = threadIdx.x; i < 2 * kHistBins / 4; i += 256) z[i] = make_uint4(0, 0, 0, 0);
}

// Standalone select: the first digit's histogram of every request's scores
// (each CTA counts its slice in shared memory and adds the non-zero bins).
__global__ void __launch_bounds__(SW_T) select_hist_kernel(SelArgs a) {
    __shared__ uint32_t h[SW_BINS];
    const int tid = threadIdx.x, lane = tid & 31;
    const int b = blockIdx.x, c = blockIdx.y;
    for (int i = tid; i < SW_BINS; i += SW_T) h[i] = 0u;
    const float* sc;
    int64_t G;
    sel_span(a, b, sc, G);
    __syncthreads();
    const int64_t pos = (int64_t)c * SW_SLICE + SW_PER * tid;
    uint32_t key[SW_PER];
    sel_load4(sc, pos, G, key);
    pdl_launch_dependents();  // the scan waits for this grid before it reads the histogram
#pragma unroll
    for (int q = 0; q < SW_PER; ++q) {
        const bool in = pos + q < G;
        const uint32_t d = key[q] >> 21;
        const unsigned m = __ballot_sync(0xffffffffu, in);
        if (in) {
            const unsigned peers = __match_any_sync(m, d);
            if (lane == __ffs(peers) - 1) atomicAdd(&h[d], (uint32_t)__popc(peers));
        }
    }
    __syncthreads();
    pdl_wait();  // the histogram block is cleared by the preceding kernel
    uint32_t* hb = a.hist + (int64_t)b * kHistBlock;
    for (int i = tid; i < SW_BINS; i += SW_T)
        if (h[i]) atomicAdd(hb + i, h[i]);
}

// ------------------------------------------------------------------ the select after the bounds
// With the tensor-core brackets of score_bound.cu, scores holds each candidate's upper bound U
// and hist the histogram of the top HB bits of the lower bounds' keys (HB = 12..14).  The bin
// b0 holding the k-th largest lower bound puts at least k exact scores at or above the bin's
// lowest value, so every candidate whose key(U) >> (32 - HB) is below b0 is out of the top k.
//  scan:  each CTA compacts its slice's candidates with key(U) >> (32 - HB) >= b0 (all of them
//         when the request has at most k) in index order and rescores them exactly in the
//         fixed chain order -- every (candidate, chain) pair a thread's work, four chains per
//         thread in flight, the chains combined per candidate in head order -- and writes
//         (exact key << 32 | index) to its region of the lists, with the count.
//  exact: SX_CTAS CTAs per batch entry; each loads every region's entries (a few hundred at
//         the 1M workload) into shared memory and ranks its share of them against all: an
//         entry with rank r < k (the number of composites above its own) goes to out[r].
//         Above SX_CAP entries (degenerate inputs, e.g. every score tied) the first CTA runs a
//         radix select over the lists instead and writes the set in index order.
// Output: the k indices ordered by (score desc, index asc) (or, above SX_CAP entries, as a
// set in index order), then -1 padding.
constexpr int SX_CAP = 4096;   // list entries the exact select ranks in shared memory
constexpr int SX_CTAS = 16;    // CTAs per batch entry of the exact select
constexpr int SX_QMAX = 16;    // index heads
constexpr int SX_SLOTS = SW_T * 4;  // chain slots of one rescoring round (four per thread)
constexpr int SB_PER = 8;              // upper bounds per thread of the bound scan
constexpr int SB_SLICE = SW_T * SB_PER;  // per bound-scan CTA: the lists region of the exact select

struct BoundSelArgs {
    SelArgs s;                 // scores = upper bounds; hist: top HB bits of the lower bounds' keys
    const uint16_t* q_idx;     // [B][Hi][128]
    const float* w_h;          // [B][Hi]
    int Hi;
    DPaged kidx;               // bf16 rows of 256 B
};

struct SxSmem {
    uint64_t ent[SX_CAP];                // composites, region by region
    alignas(16) uint32_t hist[SW_BINS];  // radix path: one digit's counts (16-byte loads)
    SwCore core;
    uint32_t pre[SW_CMAX + 1];           // exclusive prefix of the regions' entries
    uint32_t spre[SW_CMAX + 1];          // radix path: per region its selected entries, then their prefix
};
static_assert(offsetof(SxSmem, hist) % 16 == 0, "16-byte loads of the histogram");

struct SbSmem {                          // bound scan
    SwCore core;
    uint32_t cidx[SB_SLICE];             // the slice's candidates (index order)
    float qf[4 * SX_QMAX * 33];          // chain n = 4h + j: q_h[32j + d] at n * 33 + d
    float wf[SX_QMAX];
    float qv[SX_SLOTS + SW_T];           // a round's chain results, candidate c at c * (4 Hi + 1)
    uint8_t gone[SX_SLOTS / 16];         // a round's candidates whose page id is out of range
};

// The bin holding the need-th largest element of a 2^HB-bin histogram hb (global memory),
// counting from the top: thread t owns bins [top - PER + 1, top], top = 2^HB - 1 - PER t.
// Sets sm.bin (~0 when the counts hold fewer than need), sm.above and sm.cnt.
template <int HB>
__device__ __forceinline__ void sw_find_bin_wide(SwCore& sm, const uint32_t* hb, uint32_t need) {
    constexpr int PER = (1 << HB) / SW_T;
    const int top = (1 << HB) - 1 - PER * (int)threadIdx.x;
    uint32_t c[PER];
    uint32_t sum = 0;
#pragma unroll
    for (int i = 0; i < PER; i += 4) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(hb + top - PER + 1 + i));
        c[i] = v.x; c[i + 1] = v.y; c[i + 2] = v.z; c[i + 3] = v.w;
        sum += v.x + v.y + v.z + v.w;
    }
    if (threadIdx.x == 0) {
        sm.bin = ~0u;
        sm.above = 0;
        sm.cnt = 0;
    }
    uint32_t tot;
    uint32_t acc = sw_scan(sm, sum, &tot);  // its barriers order the reset
    if (sum > 0 && acc < need && need <= acc + sum) {
#pragma unroll
        for (int i = PER - 1; i >= 0; --i) {  // c[PER - 1] is bin `top`
            if (acc < need && need <= acc + c[i]) {
                sm.bin = (uint32_t)(top - (PER - 1 - i));
                sm.above = acc;
                sm.cnt = c[i];
            }
            acc += c[i];
        }
    }
    __syncthreads();
}

template <int HB>
__global__ void __launch_bounds__(SW_T, 2) select_bound_scan_kernel(BoundSelArgs a) {
    __shared__ SbSmem sm;
    const int tid = threadIdx.x;
    const int b = blockIdx.x, c = blockIdx.y, C = a.s.C, k = a.s.k;
    const float* sc;
    int64_t G;
    sel_span(a.s, b, sc, G);
    const uint32_t* hb = a.s.hist + (int64_t)b * kHistBlock;
    uint64_t* lc = a.s.lists + ((int64_t)b * C + c) * SB_SLICE;
    const bool all_in = G <= k;
    const int Hi = a.Hi, nch = 4 * Hi;
    if (!all_in) {  // the entry's query as fp32 by chain, and its weights: inputs of the step
        for (int i = tid; i < Hi * DI; i += SW_T) {
            const uint16_t v = a.q_idx[(int64_t)b * Hi * DI + i];
            const int h = i >> 7, dd = i & 127;
            sm.qf[(4 * h + (dd >> 5)) * 33 + (dd & 31)] = __uint_as_float((uint32_t)v << 16);
        }
        if (tid < Hi) sm.wf[tid] = a.w_h[(int64_t)b * Hi + tid];
    }
    pdl_wait();  // the bounds and the lower bounds' histogram come from the score kernel
    pdl_launch_dependents();

    const int64_t pos = (int64_t)c * SB_SLICE + SB_PER * tid;
    uint32_t key[SB_PER];
    sel_load4(sc, pos, G, *reinterpret_cast<uint32_t(*)[SW_PER]>(key));
    sel_load4(sc, pos + SW_PER, G, *reinterpret_cast<uint32_t(*)[SW_PER]>(key + SW_PER));
    uint32_t b0 = 0;
    if (!all_in) {
        sw_find_bin_wide<HB>(sm.core, hb, (uint32_t)k);
        b0 = sm.core.bin == ~0u ? 0u : sm.core.bin;  // (fewer than k counted cannot happen; then keep all)
    }
    uint32_t cm = 0, nc = 0;  // candidate mask over the thread's 8 scores
#pragma unroll
    for (int q = 0; q < SB_PER; ++q)
        if (pos + q < G && (all_in || (key[q] >> (32 - HB)) >= b0)) {
            cm |= 1u << q;
            ++nc;
        }
    uint32_t tot;
    uint32_t oc = sw_scan(sm.core, nc, &tot);
#pragma unroll
    for (int q = 0; q < SB_PER; ++q)
        if (cm >> q & 1u) sm.cidx[oc++] = (uint32_t)(pos + q);
    __syncthreads();
    if (all_in) {
        for (uint32_t i = tid; i < tot; i += SW_T) lc[i] = sm.cidx[i];
    } else {
        const int rc = SX_SLOTS / nch;  // candidates per round
        for (uint32_t base = 0; base < tot; base += (uint32_t)rc) {
            const int nr = (int)(tot - base < (uint32_t)rc ? tot - base : (uint32_t)rc);
            const int act = nr * nch;  // active chain slots of the round
            // chain slot tid + s * SW_T (s < 4) -> candidate slot / nch, chain slot % nch; two
            // slots in flight at a time
#pragma unroll 1
            for (int s2 = 0; s2 < 4; s2 += 2) {
                if ((tid & ~31) + s2 * SW_T >= act) break;  // (warp-uniform) no active slot left
                float p[2] = {0.f, 0.f};
                uint4 kv[2][4];
                bool ok[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int slot = tid + (s2 + u) * SW_T;
                    const uint8_t* row = nullptr;
                    if (slot < act) row = row_addr(a.kidx, b, sm.cidx[base + slot / nch], 256, a.s.status);
                    ok[u] = row != nullptr;
                    const int j = (slot % nch) & 3;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        kv[u][v] = ok[u] ? __ldg(reinterpret_cast<const uint4*>(row + 64 * j) + v) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int n = (tid + (s2 + u) * SW_T) % nch;
                    const float* qn = sm.qf + n * 33;
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const uint32_t wd[4] = {kv[u][v].x, kv[u][v].y, kv[u][v].z, kv[u][v].w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int d = 8 * v + e;
                            const float kf = (e & 1) ? bf16hi(wd[e >> 1]) : bf16lo(wd[e >> 1]);
                            p[u] = d == 0 ? __fmul_rn(qn[0], kf) : __fmaf_rn(qn[d], kf, p[u]);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int slot = tid + (s2 + u) * SW_T;
                    if (slot < act) {
                        sm.qv[(slot / nch) * (nch + 1) + slot % nch] = p[u];
                        if (slot % nch == 0) sm.gone[slot / nch] = ok[u] ? 0 : 1;
                    }
                }
            }
            __syncthreads();
            // combine: dot_h = (Q[0] + Q[2]) + (Q[1] + Q[3]), acc = fma(w_h, ReLU(dot_h), acc) in head order
            if (tid < nr) {
                const uint32_t i = base + (uint32_t)tid;
                const float* qr = sm.qv + tid * (nch + 1);
                float acc = 0.f;
                for (int h = 0; h < Hi; ++h) {
                    const float dot = (qr[4 * h] + qr[4 * h + 2]) + (qr[4 * h + 1] + qr[4 * h + 3]);
                    acc = __fmaf_rn(sm.wf[h], dot > 0.f ? dot : 0.f, acc);
                }
                if (sm.gone[tid]) acc = 0.f;  // page out of range: scored 0, as by the fixed-order kernel
                lc[i] = ((uint64_t)score_key(acc) << 32) | sm.cidx[i];
            }
            __syncthreads();
        }
    }
    if (tid == 0) a.s.counts[(int64_t)b * C + c] = tot;
}

__global__ void __launch_bounds__(SW_T, 1) select_exact_kernel(SelArgs a) {
    extern __shared__ __align__(16) uint8_t sx_raw[];
    SxSmem& sm = *reinterpret_cast<SxSmem*>(sx_raw);  // the dynamic shared memory starts 16-byte aligned
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x, part = blockIdx.y, C = a.C, k = a.k;
    const int64_t rs = a.slice;  // region stride of the lists
    const uint64_t* lb = a.lists + (int64_t)b * C * rs;
    const uint32_t* cb = a.counts + (int64_t)b * C;
    int32_t* out = a.out + (int64_t)b * k;
    pdl_wait();  // the lists and their counts come from the scan
    pdl_launch_dependents();

    uint32_t cnt[SW_PER];
#pragma unroll
    for (int j = 0; j < SW_PER; ++j) {
        const int cc = SW_PER * tid + j;
        cnt[j] = cc < C ? __ldcg(cb + cc) : 0u;
    }
    uint32_t n;
    uint32_t ex = sw_scan(sm.core, cnt[0] + cnt[1] + cnt[2] + cnt[3], &n);
#pragma unroll
    for (int j = 0; j < SW_PER; ++j) {
        const int cc = SW_PER * tid + j;
        if (cc < C) sm.pre[cc] = ex;
        ex += cnt[j];
    }
    if (tid == 0) sm.pre[C] = n;
    __syncthreads();

    if (n <= (uint32_t)SX_CAP) {
        // ---- rank every entry against all: out[rank] for rank < k.  Entry i of the concatenation
        // lies in region sw_owner(pre, i); every thread's loads go out together.
        constexpr int LPT = SX_CAP / SW_T;  // entries per thread, at most
        uint64_t ld[LPT];
#pragma unroll
        for (int q = 0; q < LPT; ++q) {
            const uint32_t i = tid + (uint32_t)q * SW_T;
            if (i < n) {
                const int cc = sw_owner(sm.pre, C, i);
                ld[q] = __ldcg(lb + (int64_t)cc * rs + (i - sm.pre[cc]));
            }
        }
#pragma unroll
        for (int q = 0; q < LPT; ++q) {
            const uint32_t i = tid + (uint32_t)q * SW_T;
            if (i < n) sm.ent[i] = sel_comp(ld[q]);
        }
        __syncthreads();
        // eight lanes per entry, each over every eighth composite, summed with shuffles
        const uint32_t per = (n + SX_CTAS - 1) / SX_CTAS;
        const uint32_t i0 = (uint32_t)part * per, i1 = i0 + per < n ? i0 + per : n;
        const uint32_t sub = (uint32_t)tid & 7u;
        for (uint32_t e0 = i0; e0 < i1; e0 += SW_T / 8) {  // (the same trip count in every lane)
            const uint32_t i = e0 + ((uint32_t)tid >> 3);
            const uint64_t v = i < i1 ? sm.ent[i] : ~0ull;
            uint32_t r = 0;
#pragma unroll 4
            for (uint32_t m = sub; m < n; m += 8) r += sm.ent[m] > v ? 1u : 0u;
            r += __shfl_xor_sync(0xffffffffu, r, 1);
            r += __shfl_xor_sync(0xffffffffu, r, 2);
            r += __shfl_xor_sync(0xffffffffu, r, 4);
            if (i < i1 && sub == 0 && r < (uint32_t)k) out[r] = (int32_t)(0x7FFFFFFFu - (uint32_t)(v & 0x7FFFFFFFu));
        }
        if (part == 0)
            for (uint32_t i = n + tid; i < (uint32_t)k; i += SW_T) out[i] = -1;
        return;
    }
    if (part != 0) return;  // (uniform per CTA)

    // ---- more entries than fit: radix select over the lists in L2, the set in index order.
    // Digits key 31..21 | 20..10 | 9..0, inverted index 30..20 | 19..10 | 9..0 (composite bits
    // 63..53 | 52..42 | 41..32 | 30..20 | 19..10 | 9..0).
    auto entry = [&](int cc, uint32_t i) -> uint64_t { return sel_comp(__ldcg(lb + (int64_t)cc * rs + i)); };
    uint64_t prefix = 0, pmask = 0;
    {
        const int shift[6] = {53, 42, 32, 20, 10, 0};
        const uint32_t dmask[6] = {2047u, 2047u, 1023u, 2047u, 1023u, 1023u};
        uint32_t need = (uint32_t)k;
        for (int dgt = 0; dgt < 6; ++dgt) {
            for (int i = tid; i < SW_BINS; i += SW_T) sm.hist[i] = 0;
            __syncthreads();
            for (int cc = warp; cc < C; cc += SW_T / 32) {
                const uint32_t m = sm.pre[cc + 1] - sm.pre[cc];
                for (uint32_t i = lane; i < m; i += 32) {
                    const uint64_t v = entry(cc, i);
                    if ((v & pmask) == prefix) atomicAdd(&sm.hist[(v >> shift[dgt]) & dmask[dgt]], 1u);
                }
            }
            __syncthreads();
            const uint4 hv = *reinterpret_cast<const uint4*>(&sm.hist[SW_BINS - 4 - 4 * tid]);
            const uint32_t h[4] = {hv.w, hv.z, hv.y, hv.x};
            sw_find_bin(sm.core, h, need);
            const uint32_t bd = sm.core.bin, above = sm.core.above, cn = sm.core.cnt;
            if (bd == ~0u) {  // inconsistent counts: cannot happen
                raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                break;
            }
            prefix |= (uint64_t)bd << shift[dgt];
            pmask |= (uint64_t)dmask[dgt] << shift[dgt];
            need -= above;
            if (cn == need) break;  // every composite of the bin is in
        }
    }
    // selected: (v & pmask) >= prefix; per region count, prefix, then write in index order
    for (int cc = warp; cc < C; cc += SW_T / 32) {
        const uint32_t m = sm.pre[cc + 1] - sm.pre[cc];
        uint32_t s = 0;
        for (uint32_t i0 = 0; i0 < m; i0 += 32) {
            const uint32_t i = i0 + lane;
            const bool f = i < m && (entry(cc, i) & pmask) >= prefix;
            s += __popc(__ballot_sync(0xffffffffu, f));
        }
        if (lane == 0) sm.spre[cc] = s;
    }
    __syncthreads();
    uint32_t v[SW_PER];
#pragma unroll
    for (int j = 0; j < SW_PER; ++j) {
        const int cc = SW_PER * tid + j;
        v[j] = cc < C ? sm.spre[cc] : 0u;
    }
    uint32_t total;
    ex = sw_scan(sm.core, v[0] + v[1] + v[2] + v[3], &total);
#pragma unroll
    for (int j = 0; j < SW_PER; ++j) {
        const int cc = SW_PER * tid + j;
        if (cc < C) sm.spre[cc] = ex;
        ex += v[j];
    }
    __syncthreads();
    for (int cc = warp; cc < C; cc += SW_T / 32) {
        const uint32_t m = sm.pre[cc + 1] - sm.pre[cc];
        uint32_t base = sm.spre[cc];
        for (uint32_t i0 = 0; i0 < m; i0 += 32) {
            const uint32_t i = i0 + lane;
            uint64_t e = 0;
            bool f = false;
            if (i < m) {
                e = entry(cc, i);
                f = (e & pmask) >= prefix;
            }
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            const uint32_t o = base + __popc(bal & ((1u << lane) - 1u));
            if (f && o < (uint32_t)k) out[o] = (int32_t)(0x7FFFFFFFu - (uint32_t)(e & 0x7FFFFFFFu));
            base += __popc(bal);
        }
    }
    if (total != (n < (uint32_t)k ? n : (uint32_t)k)) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    for (uint32_t i = total + tid; i < (uint32_t)k; i += SW_T) out[i] = -1;
}

// ------------------------------------------------------------------ host side
static int64_t select_set_ctas(int64_t max_G) { return max_G <= 0 ? 1 : (max_G + SW_SLICE - 1) / SW_SLICE; }

bool select_set_supported(int64_t max_G, int k) {
    return select_set_ctas(max_G) <= SW_CMAX && k >= 1 && k <= 2048;
}

static int64_t bound_scan_ctas(int64_t max_G) { return max_G <= 0 ? 1 : (max_G + SB_SLICE - 1) / SB_SLICE; }

size_t select_set_lists_bytes(int B, int64_t max_G) {
    if (!select_set_supported(max_G, 1)) return 0;
    const int64_t C = select_set_ctas(max_G), Cb = bound_scan_ctas(max_G);  // (either select's layout)
    const size_t wide = align_up((size_t)B * C * SW_SLICE * sizeof(uint64_t), 256) +
                        align_up((size_t)B * C * sizeof(uint32_t), 256);
    const size_t bound = align_up((size_t)B * Cb * SB_SLICE * sizeof(uint64_t), 256) +
                         align_up((size_t)B * Cb * sizeof(uint32_t), 256);
    return wide > bound ? wide : bound;
}

cudaError_t launch_select_set(const SelectSetLaunch& h, cudaStream_t s, bool pdl) {
    SelArgs a;
    a.scores = h.scores;
    a.score_stride = h.score_stride;
    a.n_tokens = h.n_tokens;
    a.nq = h.nq > 1 ? h.nq : 1;
    a.ratio = h.ratio;
    a.offsets = h.offsets;
    a.G = h.G;
    a.sorted = h.standalone ? 1 : 0;
    a.keys_out = h.keys_out;
    a.C = (int)select_set_ctas(h.max_G);
    a.k = h.k;
    a.out = h.idx_out;
    a.hist = h.hist;
    a.lists = reinterpret_cast<uint64_t*>(h.lists);
    a.counts = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(h.lists) +
                                           align_up((size_t)h.B * a.C * SW_SLICE * sizeof(uint64_t), 256));
    a.slice = SW_SLICE;
    a.status = h.status;
    const size_t smem = sizeof(SwFinSmem);
    static_assert(sizeof(SwFinSmem) + SW_SCAN_SPREAD_SMEM + 2 * 1024 <= 228 * 1024, "a scan and a finish CTA share an SM");
    {
        cudaError_t e = set_func_attr_once((const void*)select_finish_kernel<88>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = set_func_attr_once((const void*)select_finish_kernel<64>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e == cudaSuccess)
            e = set_func_attr_once((const void*)select_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SW_SCAN_SPREAD_SMEM);
        if (e == cudaSuccess)
            e = set_func_attr_once((const void*)select_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SW_SCAN_SPREAD_SMEM);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int sms = device_sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    // grid (request, region): the blocks are dispatched region-major, so a batch's region 0s
    // (which carry the finish's general path) are all in the first wave
    cfg.gridDim = dim3((unsigned)h.B, (unsigned)a.C, 1);
    cfg.blockDim = dim3(SW_T, 1, 1);
    // one scan CTA per SM when the grid fits on the SMs; a larger grid is packed instead, so
    // that it stays one wave
    cfg.dynamicSmemBytes = (int64_t)a.C * h.B <= sms ? SW_SCAN_SPREAD_SMEM : 0;
    cfg.stream = s;
    cudaError_t e = cudaSuccess;
    if (h.standalone) {  // histograms cleared, first digit counted; the scan follows programmatically
        cudaLaunchConfig_t z = {};
        z.gridDim = dim3((unsigned)h.B, 1, 1);
        z.blockDim = dim3(256, 1, 1);
        z.stream = s;
        e = cudaLaunchKernelEx(&z, select_zero_kernel, h.hist);
        if (e != cudaSuccess) return e;
        e = cudaLaunchKernelEx(&cfg, select_hist_kernel, a);
        if (e != cudaSuccess) return e;
    }
    e = cudaLaunchKernelEx(&cfg, select_scan_kernel, a);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem;
    const int64_t ctas = (int64_t)h.B * a.C;
    return ctas > sms && ctas <= 2LL * sms ? cudaLaunchKernelEx(&cfg, select_finish_kernel<64>, a)
                                           : cudaLaunchKernelEx(&cfg, select_finish_kernel<88>, a);
}

cudaError_t launch_select_bound(const SelectSetLaunch& h, const BoundRescore& r, cudaStream_t s, bool pdl) {
    if (!h.n_tokens || h.standalone || r.Hi < 1 || r.Hi > SX_QMAX) return cudaErrorInvalidValue;
    BoundSelArgs a;
    a.s.scores = h.scores;
    a.s.score_stride = h.score_stride;
    a.s.n_tokens = h.n_tokens;
    a.s.nq = h.nq > 1 ? h.nq : 1;
    a.s.ratio = h.ratio;
    a.s.offsets = nullptr;
    a.s.G = 0;
    a.s.sorted = 0;
    a.s.keys_out = nullptr;
    a.s.C = (int)bound_scan_ctas(h.max_G);
    a.s.k = h.k;
    a.s.out = h.idx_out;
    a.s.hist = h.hist;
    a.s.lists = reinterpret_cast<uint64_t*>(h.lists);
    a.s.counts = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(h.lists) +
                                             align_up((size_t)h.B * a.s.C * SB_SLICE * sizeof(uint64_t), 256));
    a.s.slice = SB_SLICE;
    a.s.status = h.status;
    a.q_idx = static_cast<const uint16_t*>(r.q_idx);
    a.w_h = r.w_h;
    a.Hi = r.Hi;
    a.kidx.base = static_cast<const uint8_t*>(r.kidx.base);
    a.kidx.pt = r.kidx.pt;
    a.kidx.pt_stride = r.kidx.pt_stride;
    a.kidx.page_stride = r.kidx.page_stride;
    a.kidx.n_pages = r.kidx.n_pages;
    a.kidx.rpp = r.kidx.rpp;
    a.kidx.qpr = h.nq > 1 ? h.nq : 1;
    const size_t smem = sizeof(SxSmem);
    const int hbits = bound_hist_bits(a.s.nq);
    const void* scan = hbits == 14 ? (const void*)select_bound_scan_kernel<14>
                     : hbits == 13 ? (const void*)select_bound_scan_kernel<13>
                                   : (const void*)select_bound_scan_kernel<12>;
    {
        cudaError_t e = set_func_attr_once((const void*)select_exact_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const int sms = device_sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    cfg.gridDim = dim3((unsigned)h.B, (unsigned)a.s.C, 1);
    cfg.blockDim = dim3(SW_T, 1, 1);
    cfg.dynamicSmemBytes = 0;  // two scan CTAs per SM: 4 x 64 slices of the 1M workload are one wave
    cfg.stream = s;
    void* args[] = {&a};
    cudaError_t e = cudaLaunchKernelExC(&cfg, scan, args);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)h.B, (unsigned)SX_CTAS, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.numAttrs = 1;  // waits for the scan (griddepcontrol.wait)
    return cudaLaunchKernelEx(&cfg, select_exact_kernel, a.s);
}

}  // namespace csa
