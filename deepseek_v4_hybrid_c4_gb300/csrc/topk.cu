// Stage 3: exact top-k of the index scores by radix select ("SGLang 如何为 DeepSeek V4
// 打造「Day-0」推理加速", sec. "创新 2", Lightning TopK: per-CTA histograms reduced
// to a threshold tau, then a scatter of the entries above tau; "DeepSeek-V4 本地部署，
// SGLang 把活做絕了", sec. "Kernel 層一堆狠活").
//
// Order: descending order-preserving 32-bit key of the fp32 score, ties to the lower
// index.  Equivalently, descending 63-bit composite V = key << 31 | (2^31 - 1 - index),
// which is unique per element, so the selected set and its order are unique.  Digits
// of V, high to low: key bits 31..21 | 20..10 | 9..0, then inverted-index bits
// 30..20 | 19..10 | 9..0.
//
// Wide select, two phases in one launch with grid (C, B):
//  A. Every CTA of request b reads the first digit's histogram of the whole request
//     (fused into the score kernel in the decode step; built by topk_hist_kernel for
//     the standalone call, per-CTA histograms summed inside a cluster of 8 through
//     distributed shared memory) and finds the bin b0 holding the k-th key.  It scans
//     its slice of the scores once: keys above b0 are winners, keys in b0 survivors,
//     both appended to global lists with one atomic per warp.
//  B. The last CTA of the request to finish (a completion counter; no CTA waits for
//     another) loads both lists into shared memory and refines the survivors digit by
//     digit (histogram, bin of the remaining need, compaction) until winners plus
//     survivors fit one sort; then a bitonic sort by V gives the k outputs in order.
//     If more survivors arrive than the list holds, the digits run over the scores in
//     global memory until the candidates fit.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int TK_T = 1024;           // threads per CTA
constexpr int TK_BINS = kHistBins;   // 2048: widest digit
constexpr int TK_KMAX = 2048;        // largest k; winners list capacity
constexpr int TK_SCAP = 16384;       // survivors held in shared memory
constexpr int TK_MAXC = 64;          // most select CTAs per request
constexpr int TK_CHUNK = 4 * TK_T;   // scores per CTA in phase A (one float4 per thread)
constexpr int TK_HCL = 8;            // cluster size of the standalone histogram kernel
constexpr int TK_HCHUNK = 8 * TK_T;  // scores per CTA of the histogram kernel

struct TopkArgs {
    const float* scores;
    int B;
    int64_t G;
    const int64_t* offsets;
    const int64_t* n_tokens;
    int ratio;
    int64_t score_stride;
    int k;
    int32_t* idx_out;
    uint32_t* keys_out;
    int sorted;       // 1: output ordered by (score desc, index asc); 0: the set, in a fixed order
    uint32_t* hist;   // [B][kHistBlock]: digit histograms, control words, per-CTA counts
    uint2* wlist;     // [B][C][capw] winners {key, index}, one region per CTA
    uint2* slist;     // [B][C][caps] survivors
    int64_t capw, caps;
    int32_t* status;
};

struct TkSmem {
    uint32_t hist[TK_BINS];
    uint32_t okey[TK_KMAX];     // winners, then the union to sort
    int32_t oidx[TK_KMAX];
    uint32_t ckey[TK_SCAP];     // survivors
    int32_t cidx[TK_SCAP];
    uint64_t sortbuf[TK_KMAX];
    uint32_t wsum[32];
    uint32_t xoff[32];
    uint32_t pw[TK_MAXC + 1], ps[TK_MAXC + 1];  // per-CTA list offsets (phase B)
    int n_sel, n_cand, n_new;
    uint32_t bin, above, cnt, last;
};

__device__ __forceinline__ void request_span(const TopkArgs& a, int b, const float*& sc, int64_t& G) {
    if (a.offsets) {
        const int64_t o0 = a.offsets[b], o1 = a.offsets[b + 1];
        sc = a.scores + o0;
        G = o1 - o0;
    } else if (a.n_tokens) {
        sc = a.scores + (int64_t)b * a.score_stride;
        G = a.n_tokens[b] / a.ratio;
    } else {
        sc = a.scores;
        G = a.G;
    }
    if (G < 0) G = 0;
}

__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t digit, bool active) {
    const unsigned m = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(m, digit);
    if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
}

// Exclusive block scan of v over TK_T threads; returns the prefix, *total = sum.
__device__ __forceinline__ uint32_t block_scan(TkSmem& sm, uint32_t v, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = sm.wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        sm.wsum[lane] = w;  // inclusive prefix of warp totals
    }
    __syncthreads();
    const uint32_t before = warp ? sm.wsum[warp - 1] : 0u;
    *total = sm.wsum[31];
    __syncthreads();
    return before + x - v;
}

// Order-preserving split of one chunk (one element per thread): `win` elements are
// appended to the winners (sm.n_sel), `stay` elements to the survivors at *n_stay, both
// in thread order.  Returns this thread's slots (-1 when not taken).  Every thread calls it.
__device__ __forceinline__ void ordered_split(TkSmem& sm, bool win, bool stay, int* n_stay, int& so, int& sc) {
    uint32_t tot;
    const uint32_t ex = block_scan(sm, (win ? 0x10000u : 0u) | (stay ? 1u : 0u), &tot);
    so = win ? sm.n_sel + (int)(ex >> 16) : -1;
    sc = stay ? *n_stay + (int)(ex & 0xFFFFu) : -1;
    __syncthreads();  // every thread has read the counters
    if (threadIdx.x == 0) {
        sm.n_sel += (int)(tot >> 16);
        *n_stay += (int)(tot & 0xFFFFu);
    }
    __syncthreads();
}

// The bin holding the need-th largest element counted from the top bin, given this
// thread's two bins' counts (bins nbins-1-2t and nbins-2-2t, high first).  Writes sm.bin,
// sm.above (count in higher bins) and sm.cnt (count in the bin).
__device__ __forceinline__ void find_bin_vals(TkSmem& sm, uint32_t th, uint32_t tl, int nbins, uint32_t need) {
    const int t = threadIdx.x;
    const int bh = nbins - 1 - 2 * t, bl = nbins - 2 - 2 * t;
    if (t == 0) {
        sm.bin = 0;
        sm.above = 0;
        sm.cnt = 0;
    }
    uint32_t total;
    const uint32_t excl = block_scan(sm, th + tl, &total);
    if (bl >= 0) {
        if (th > 0 && excl < need && need <= excl + th) {
            sm.bin = (uint32_t)bh;
            sm.above = excl;
            sm.cnt = th;
        } else if (tl > 0 && excl + th < need && need <= excl + th + tl) {
            sm.bin = (uint32_t)bl;
            sm.above = excl + th;
            sm.cnt = tl;
        }
    }
    __syncthreads();
}
// From a histogram in global memory written by an earlier kernel (read-only path).
__device__ __forceinline__ void find_bin_global(TkSmem& sm, const uint32_t* gh, int nbins, uint32_t need) {
    const int bh = nbins - 1 - 2 * (int)threadIdx.x, bl = bh - 1;
    const uint32_t th = bl >= 0 ? __ldg(gh + bh) : 0u, tl = bl >= 0 ? __ldg(gh + bl) : 0u;
    find_bin_vals(sm, th, tl, nbins, need);
}
// From this CTA's sm.hist.
__device__ __forceinline__ void find_bin_local(TkSmem& sm, int nbins, uint32_t need) {
    const int bh = nbins - 1 - 2 * (int)threadIdx.x, bl = bh - 1;
    const uint32_t th = bl >= 0 ? sm.hist[bh] : 0u, tl = bl >= 0 ? sm.hist[bl] : 0u;
    find_bin_vals(sm, th, tl, nbins, need);
}

// The keys of 4 consecutive scores pos .. pos+3 (a float4 load when the whole group is
// in range and 16-byte aligned); out-of-range entries read as key 0.
__device__ __forceinline__ void load4(const float* sc, int64_t pos, int64_t hi, bool vec, uint32_t (&key)[4]) {
    float v[4];
    if (vec && pos + 3 < hi) {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(sc + pos));
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[q] = pos + q < hi ? __ldcg(sc + pos + q) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) key[q] = score_key(v[q]);
}

// Bitonic sort of the 64 composites of a warp, two per lane (element 2*lane + r), larger
// first: the stride-1 stages stay in the lane, the others use shuffles.
__device__ __forceinline__ void warp_sort64(uint64_t (&v)[2]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
        for (int j = size >> 1; j > 0; j >>= 1) {
            if (j == 1) {
                const bool desc = ((2 * lane) & size) == 0;
                const uint64_t mx = v[0] > v[1] ? v[0] : v[1], mn = v[0] > v[1] ? v[1] : v[0];
                v[0] = desc ? mx : mn;
                v[1] = desc ? mn : mx;
            } else {
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const uint64_t pv = __shfl_xor_sync(0xffffffffu, v[r], j >> 1);
                    const int i = 2 * lane + r;
                    const bool lower = (i & j) == 0, desc = (i & size) == 0;
                    const uint64_t mx = v[r] > pv ? v[r] : pv, mn = v[r] > pv ? pv : v[r];
                    v[r] = (desc == lower) ? mx : mn;
                }
            }
        }
    }
}

// Order okey/oidx[0..total) (total <= TK_KMAX) by (key desc, index asc) and write the
// first k (then -1 padding).  Warp w sorts elements [64w, 64w+64) into a run; an
// element's output position is its place in its own run plus, for every other run, the
// number of that run's elements above it (binary search).  Composites are unique and
// the zero padding sits below every element, so the positions are exact.
__device__ void rank_scatter(TkSmem& sm, int total, int k, int32_t* out, uint32_t* kout) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (total > TK_KMAX) total = TK_KMAX;
    const int nruns = (total + 63) / 64;
    uint64_t v[2] = {0ull, 0ull};
    uint64_t* runs = sm.sortbuf;
    if (warp < nruns) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int i = 64 * warp + 2 * lane + r;
            // composite: key << 32 | (2^31 - 1 - index); 0 = padding
            v[r] = i < total ? ((uint64_t)sm.okey[i] << 32) | (uint32_t)(0x7FFFFFFF - sm.oidx[i]) : 0ull;
        }
        warp_sort64(v);
        runs[64 * warp + 2 * lane] = v[0];
        runs[64 * warp + 2 * lane + 1] = v[1];
    }
    __syncthreads();
    if (warp < nruns) {
        int rank[2] = {2 * lane, 2 * lane + 1};
        for (int o = 0; o < nruns; ++o) {
            if (o == warp) continue;
            const uint64_t* run = runs + 64 * o;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                int lo = 0;  // elements of run o above v[r]: the run is sorted larger first
#pragma unroll
                for (int step = 32; step > 0; step >>= 1)
                    if (run[lo + step - 1] > v[r]) lo += step;
                if (lo == 63 && run[63] > v[r]) lo = 64;
                rank[r] += lo;
            }
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (v[r] != 0ull && rank[r] < k) {
                out[rank[r]] = (int32_t)(0x7FFFFFFF - (uint32_t)v[r]);
                if (kout) kout[rank[r]] = (uint32_t)(v[r] >> 32);
            }
        }
    }
    for (int i = total + tid; i < k; i += TK_T) {
        out[i] = -1;
        if (kout) kout[i] = 0u;
    }
}

// Digit d (1..5) of the composite V of (key, index); see the header.
__device__ __forceinline__ uint32_t digit_of(int d, uint32_t key, int32_t idx) {
    const uint32_t inv = 0x7FFFFFFFu - (uint32_t)idx;
    switch (d) {
        case 1: return (key >> 10) & 2047u;
        case 2: return key & 1023u;
        case 3: return (inv >> 20) & 2047u;
        case 4: return (inv >> 10) & 1023u;
        default: return inv & 1023u;
    }
}
__device__ __forceinline__ int digit_bins(int d) { return (d == 1 || d == 3) ? 2048 : 1024; }

// Standalone first digit: the histogram of key >> 21 over every request's scores.  Each
// CTA counts its slice in shared memory; the cluster's rank-0 CTA sums the 8 CTAs'
// histograms through distributed shared memory and adds the non-zero bins to the global
// histogram (zeroed beforehand).
__global__ void __launch_bounds__(TK_T, 1) topk_hist_kernel(TopkArgs a) {
    __shared__ uint32_t h[TK_BINS];
    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const float* sc;
    int64_t G;
    request_span(a, b, sc, G);
    for (int i = tid; i < TK_BINS; i += TK_T) h[i] = 0;
    __syncthreads();
    const int64_t lo = min((int64_t)blockIdx.x * TK_HCHUNK, G), hi = min(lo + TK_HCHUNK, G);
    const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
    for (int64_t base = lo; base < hi; base += 4 * TK_T) {  // the same trip count for every thread
        const int64_t pos = base + 4 * tid;
        uint32_t key[4];
        load4(sc, pos, hi, vec, key);
#pragma unroll
        for (int q = 0; q < 4; ++q) hist_add(h, key[q] >> 21, pos + q < hi);
    }
    cluster_sync();
    if (cluster_ctarank() == 0) {
        uint32_t* gh = a.hist + (int64_t)b * kHistBlock;
        for (int i = tid; i < TK_BINS; i += TK_T) {
            const uint32_t ai = smem_u32(&h[i]);
            uint32_t v = 0;
#pragma unroll
            for (int c = 0; c < TK_HCL; ++c) v += ld_dsmem_u32(mapa(ai, c));
            if (v) atomicAdd(gh + i, v);
        }
    }
    cluster_sync();  // the other CTAs' shared memory stays alive until it has been read
}

// prefix match of (key, index) on digits 0 .. d-1
__device__ __forceinline__ bool prefix_match(const uint32_t (&bins)[6], int d, uint32_t key, int32_t idx) {
    if ((key >> 21) != bins[0]) return false;
    for (int e = 1; e < d; ++e)
        if (digit_of(e, key, idx) != bins[e]) return false;
    return true;
}

__global__ void __launch_bounds__(TK_T, 1) topk_select_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();               // scores (and the fused histogram) come from the preceding kernel
    pdl_launch_dependents();
    const int b = blockIdx.y;
    const int C = (int)gridDim.x;
    const float* sc;
    int64_t G;
    request_span(a, b, sc, G);
    const int k = a.k;
    uint32_t* ghist = a.hist + (int64_t)b * kHistBlock;   // first digit (key bits 31..21)
    uint32_t* ghist1 = ghist + kHistBins;                 // second digit of the survivors
    uint32_t* ctl = ghist + 2 * kHistBins;                // [0] finished CTAs
    uint32_t* table = ctl + 32;                           // [c] = {winners, survivors} of CTA c
    int32_t* out = a.idx_out + (int64_t)b * k;
    uint32_t* kout = a.keys_out ? a.keys_out + (int64_t)b * k : nullptr;
    const bool all_in = G <= k;  // every candidate is selected
    const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15) == 0;

    // ---- A. one scan of this CTA's slice: winners (first digit above b0) and survivors
    //      (= b0) compacted, in index order, into this CTA's own list regions
    const int64_t chunk = (((G + C - 1) / C) + 3) & ~int64_t(3);
    const int64_t lo = min((int64_t)blockIdx.x * chunk, G), hi = min(lo + chunk, G);
    uint2* wl = a.wlist + ((int64_t)b * C + blockIdx.x) * a.capw;
    uint2* sl = a.slist + ((int64_t)b * C + blockIdx.x) * a.caps;
    uint32_t key[4];
    load4(sc, lo + 4 * tid, hi, vec, key);  // in flight while the threshold bin is found
    for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[i] = 0;
    uint32_t b0 = 0;
    if (!all_in) {
        find_bin_global(sm, ghist, TK_BINS, (uint32_t)k);
        b0 = sm.bin;
    } else {
        __syncthreads();
    }
    uint32_t run_w = 0, run_s = 0;  // this CTA's list lengths so far
    for (int64_t base = lo; base < hi; base += TK_CHUNK) {
        const int64_t pos = base + 4 * tid;
        if (base != lo) load4(sc, pos, hi, vec, key);
        uint32_t ns = 0, nc = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = pos + q < hi;
            const uint32_t d = key[q] >> 21;
            ns += (in && (all_in || d > b0)) ? 1u : 0u;
            nc += (in && !all_in && d == b0) ? 1u : 0u;
        }
        // CTA-wide exclusive offsets (16-bit halves: at most TK_CHUNK per pass)
        const uint32_t v = (ns << 16) | nc;
        uint32_t x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) sm.wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            const uint32_t w = sm.wsum[lane];
            uint32_t wx = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, wx, o);
                if (lane >= o) wx += y;
            }
            sm.xoff[lane] = wx - w;
            if (lane == 31) sm.cnt = wx;
        }
        __syncthreads();
        const uint32_t ex = sm.xoff[warp] + (x - v), tot = sm.cnt;
        uint32_t bs = run_w + (ex >> 16), bc = run_s + (ex & 0xFFFFu);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = pos + q < hi;
            const uint32_t d = key[q] >> 21;
            const bool win = in && (all_in || d > b0), sur = in && !all_in && d == b0;
            if (win) {
                if (bs < (uint32_t)a.capw) wl[bs] = make_uint2(key[q], (uint32_t)(pos + q));
                else raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                ++bs;
            } else if (sur) {
                if (bc < (uint32_t)a.caps) sl[bc] = make_uint2(key[q], (uint32_t)(pos + q));
                ++bc;  // past the capacity only counted: phase B then scans the scores instead
            }
            hist_add(sm.hist, (key[q] >> 10) & 2047u, sur);  // the survivors' second digit
        }
        run_w += tot >> 16;
        run_s += tot & 0xFFFFu;
        __syncthreads();
    }
    if (tid == 0) {
        table[2 * blockIdx.x] = min(run_w, (uint32_t)a.capw);
        table[2 * blockIdx.x + 1] = run_s;
    }
    for (int i = tid; i < TK_BINS; i += TK_T) {
        const uint32_t c = sm.hist[i];
        if (c) atomicAdd(ghist1 + i, c);
    }
    // ---- the last CTA of the request to finish goes on (every thread's list entries and
    //      counts are made visible before the CTA counts itself finished)
    __threadfence();
    __syncthreads();
    if (tid == 0) sm.last = atomicAdd(&ctl[0], 1u) == (uint32_t)C - 1 ? 1u : 0u;
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    // ---- B. gather the lists, refine the survivors digit by digit, rank the union
    // the second digit's histogram bins of this thread, loaded early (L2: written by this grid)
    const int bh = TK_BINS - 1 - 2 * tid, bl = bh - 1;
    const uint32_t h1h = __ldcg(ghist1 + bh), h1l = __ldcg(ghist1 + bl);
    if (warp == 0) {  // per-CTA list offsets: exclusive prefix over the table
        uint32_t cw = 0, cs = 0;
        bool over = false;
        for (int c0 = 0; c0 < C; c0 += 32) {
            const int c = c0 + lane;
            const uint32_t tw = c < C ? __ldcg(table + 2 * c) : 0u, ts = c < C ? __ldcg(table + 2 * c + 1) : 0u;
            over |= __any_sync(0xffffffffu, ts > (uint32_t)a.caps);
            uint32_t xw = tw, xs = ts;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t yw = __shfl_up_sync(0xffffffffu, xw, o), ys = __shfl_up_sync(0xffffffffu, xs, o);
                if (lane >= o) { xw += yw; xs += ys; }
            }
            if (c < C) {
                sm.pw[c] = cw + xw - tw;
                sm.ps[c] = cs + xs - ts;
            }
            cw += __shfl_sync(0xffffffffu, xw, 31);
            cs += __shfl_sync(0xffffffffu, xs, 31);
        }
        if (lane == 0) {
            sm.pw[C] = cw;
            sm.ps[C] = cs;
            sm.n_new = over ? 1 : 0;  // a CTA's survivors overflowed its region
        }
    }
    __syncthreads();
    const int n_w0 = (int)min(sm.pw[C], (uint32_t)TK_KMAX), n_s0 = (int)sm.ps[C];
    // element j of the concatenated lists: its CTA by binary search over the prefixes
    auto region = [&](const uint32_t* pre, uint32_t j) {
        int r = 0;
        for (int step = TK_MAXC / 2; step > 0; step >>= 1)
            if (r + step <= C - 1 && pre[r + step] <= j) r += step;
        return r;
    };
    const uint2* wl0 = a.wlist + (int64_t)b * C * a.capw;
    const uint2* sl0 = a.slist + (int64_t)b * C * a.caps;
    for (int j = tid; j < n_w0; j += TK_T) {
        const int r = region(sm.pw, (uint32_t)j);
        const uint2 e = __ldcg(wl0 + (int64_t)r * a.capw + (j - (int)sm.pw[r]));
        sm.okey[j] = e.x;
        sm.oidx[j] = (int32_t)e.y;
    }
    const bool s_fit = n_s0 <= TK_SCAP && sm.n_new == 0;
    if (!all_in && s_fit) {
#pragma unroll 4
        for (int j = tid; j < n_s0; j += TK_T) {
            const int r = region(sm.ps, (uint32_t)j);
            const uint2 e = __ldcg(sl0 + (int64_t)r * a.caps + (j - (int)sm.ps[r]));
            sm.ckey[j] = e.x;
            sm.cidx[j] = (int32_t)e.y;
        }
    }
    if (tid == 0) {
        sm.n_sel = n_w0;
        sm.n_cand = all_in ? 0 : n_s0;
    }
    __syncthreads();
    uint32_t need = all_in ? 0u : (uint32_t)k - (uint32_t)n_w0;
    // refine until winners plus survivors fit one ranking (sorted output) or are exactly the
    // k selected (set output: the survivors left are then exactly the ones needed)
    const int rank_max = a.sorted ? (k <= 1024 ? 1024 : TK_KMAX) : k;
    uint32_t bins[6] = {b0, 0, 0, 0, 0, 0};
    bool implicit = !all_in && !s_fit;  // survivors not in shared memory: the digits scan the scores
    for (int d = 1; d <= 5 && sm.n_sel + sm.n_cand > rank_max; ++d) {
        const int nb = digit_bins(d);
        if (d == 1) {
            find_bin_vals(sm, h1h, h1l, TK_BINS, need);  // counted by phase A
        } else {
            for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[i] = 0;
            __syncthreads();
            if (!implicit) {
                const int n = sm.n_cand;
                for (int i0 = 0; i0 < n; i0 += TK_T) {
                    const int i = i0 + tid;
                    const bool in = i < n;
                    hist_add(sm.hist, in ? digit_of(d, sm.ckey[i], sm.cidx[i]) : 0u, in);
                }
            } else {
                for (int64_t p0 = 0; p0 < G; p0 += 4 * TK_T) {
                    uint32_t kk[4];
                    const int64_t pos = p0 + 4 * tid;
                    load4(sc, pos, G, vec, kk);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int32_t idx = (int32_t)(pos + q);
                        const bool in = pos + q < G && prefix_match(bins, d, kk[q], idx);
                        hist_add(sm.hist, in ? digit_of(d, kk[q], idx) : 0u, in);
                    }
                }
            }
            __syncthreads();
            find_bin_local(sm, nb, need);
        }
        const uint32_t dbin = sm.bin, d_n = sm.cnt;
        need -= sm.above;
        bins[d] = dbin;
        if (!implicit) {
            // in-place compaction: a chunk is read by everyone before any of it is overwritten
            const int n = sm.n_cand;
            if (tid == 0) sm.n_new = 0;
            __syncthreads();
            for (int i0 = 0; i0 < n; i0 += TK_T) {
                const int i = i0 + tid;
                const bool in = i < n;
                const uint32_t kk = in ? sm.ckey[i] : 0u;
                const int32_t idx = in ? sm.cidx[i] : 0;
                __syncthreads();
                const uint32_t dv = digit_of(d, kk, idx);
                int so, c;
                ordered_split(sm, in && dv > dbin, in && dv == dbin, &sm.n_new, so, c);
                if (so >= 0 && so < TK_KMAX) { sm.okey[so] = kk; sm.oidx[so] = idx; }
                if (c >= 0) { sm.ckey[c] = kk; sm.cidx[c] = idx; }
            }
            __syncthreads();
            if (tid == 0) sm.n_cand = sm.n_new;
        } else {
            const bool g2 = d_n <= (uint32_t)TK_SCAP;
            if (tid == 0) sm.n_cand = 0;
            __syncthreads();
            for (int64_t p0 = 0; p0 < G; p0 += 4 * TK_T) {
                uint32_t kk[4];
                const int64_t pos = p0 + 4 * tid;
                load4(sc, pos, G, vec, kk);
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // a fixed order: element q of every thread, by thread
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < G && prefix_match(bins, d, kk[q], idx);
                    const uint32_t dv = digit_of(d, kk[q], idx);
                    int so, c;
                    ordered_split(sm, in && dv > dbin, g2 && in && dv == dbin, &sm.n_cand, so, c);
                    if (so >= 0 && so < TK_KMAX) { sm.okey[so] = kk[q]; sm.oidx[so] = idx; }
                    if (c >= 0 && c < TK_SCAP) { sm.ckey[c] = kk[q]; sm.cidx[c] = idx; }
                }
            }
            __syncthreads();
            if (tid == 0 && !g2) sm.n_cand = (int)d_n;
            implicit = !g2;
        }
        __syncthreads();
    }
    // ---- the union of winners and survivors fits one ranking
    const int n_w = sm.n_sel, n_c = implicit ? 0 : sm.n_cand;
    if (tid == 0 && n_w + n_c > TK_KMAX) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    for (int i = tid; i < n_c && n_w + i < TK_KMAX; i += TK_T) {
        sm.okey[n_w + i] = sm.ckey[i];
        sm.oidx[n_w + i] = sm.cidx[i];
    }
    __syncthreads();
    if (a.sorted) {
        rank_scatter(sm, min(n_w + n_c, TK_KMAX), k, out, kout);
    } else {  // the set in its fixed order: winners by round, then the last survivors
        const int tot = min(n_w + n_c, k);
        for (int i = tid; i < k; i += TK_T) {
            out[i] = i < tot ? sm.oidx[i] : -1;
            if (kout) kout[i] = i < tot ? sm.okey[i] : 0u;
        }
    }
    if (tid == 0) ctl[0] = 0u;  // the counter is ready for the next call on this workspace
}

// Phase-A CTAs per request and the per-CTA list capacities for a batch bound max_G.
// Winners: a CTA never holds more than min(slice, k).  Survivors: an even share of what
// phase B can hold in shared memory (at least 256); a CTA with more only counts them and
// phase B then works from the scores.
struct TopkGeometry {
    int C;
    int64_t capw, caps;
};
static TopkGeometry topk_geometry(int64_t max_G, int k) {
    TopkGeometry g;
    int64_t c = (max_G + TK_CHUNK - 1) / TK_CHUNK;
    if (c > TK_MAXC) c = TK_MAXC;
    if (c < 1) c = 1;
    g.C = (int)c;
    const int64_t slice = ((((max_G + c - 1) / c) + 3) & ~int64_t(3));
    int64_t share = TK_SCAP / c;
    if (share < 256) share = 256;
    g.caps = slice < share ? slice : share;
    if (g.caps < 4) g.caps = 4;
    g.capw = slice < k ? slice : k;
    if (g.capw < 4) g.capw = 4;
    return g;
}

size_t topk_lists_bytes(int B, int64_t max_G, int k) {
    const TopkGeometry g = topk_geometry(max_G, k);
    return (size_t)B * g.C * (size_t)(g.capw + g.caps) * sizeof(uint2);
}

static TopkArgs topk_args(const TopkLaunch& h) {
    const TopkGeometry g = topk_geometry(h.max_G, h.k);
    TopkArgs a;
    a.scores = h.scores;
    a.B = h.B;
    a.G = h.G;
    a.offsets = h.offsets;
    a.n_tokens = h.n_tokens;
    a.ratio = h.ratio;
    a.score_stride = h.score_stride;
    a.k = h.k;
    a.idx_out = h.idx_out;
    a.keys_out = h.keys_out;
    a.sorted = h.sorted ? 1 : 0;
    a.hist = h.hist;
    a.capw = g.capw;
    a.caps = g.caps;
    a.wlist = reinterpret_cast<uint2*>(h.lists);
    a.slist = reinterpret_cast<uint2*>(h.lists) + (size_t)h.B * g.C * g.capw;
    a.status = h.status;
    return a;
}

cudaError_t launch_topk_hist(const TopkLaunch& h, cudaStream_t s) {
    const TopkArgs a = topk_args(h);
    int64_t per = (h.max_G + TK_HCHUNK - 1) / TK_HCHUNK;
    per = (per + TK_HCL - 1) / TK_HCL * TK_HCL;
    if (per < TK_HCL) per = TK_HCL;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = TK_HCL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3((unsigned)per, (unsigned)h.B, 1);
    cfg.blockDim = dim3(TK_T, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, topk_hist_kernel, a);
}

cudaError_t launch_topk(const TopkLaunch& h, cudaStream_t s, bool pdl) {
    const TopkArgs a = topk_args(h);
    const size_t smem = sizeof(TkSmem);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((unsigned)topk_geometry(h.max_G, h.k).C, (unsigned)h.B, 1);
    cfg.blockDim = dim3(TK_T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, topk_select_kernel, a);
}

}  // namespace csa
