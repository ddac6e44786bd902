// Stage 3: exact top-k of the index scores by cluster radix select ("SGLang 如何为
// DeepSeek V4 打造「Day-0」推理加速", sec. "创新 2", Lightning TopK: a cluster of CTAs,
// per-CTA histograms reduced inside the cluster to a threshold tau, then a scatter of the
// entries above tau; "DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "Kernel 層一堆狠活").
//
// Order: descending order-preserving 32-bit key of the fp32 score, ties to the lower
// index.  Equivalently, descending 63-bit composite V = key << 31 | (2^31 - 1 - index),
// which is unique per element, so the selected set and its order are unique.  Digits of
// V, high to low: key bits 31..21 | 20..10 | 9..0, then inverted-index bits 30..20 |
// 19..10 | 9..0.
//
// One thread-block cluster of CL <= 16 CTAs per request; CTA r owns the contiguous slice
// r of the scores and keeps everything about it in its own shared memory:
//  1. The first digit's histogram of the whole request -- fused into the score kernel in
//     the decode step (read from global memory), otherwise counted per CTA and summed the
//     same way as the rounds -- gives the bin b0 holding the k-th key.
//  2. One scan of the slice: keys above b0 are winners, keys in b0 survivors, each list
//     compacted in index order (block-wide prefix sums, no atomics).
//  3. Rounds over the next digits: each CTA counts its survivors' digit in its own shared
//     memory; after one cluster barrier every CTA sums every CTA's counts of its bins through
//     distributed shared memory (the reduction inside the cluster) and finds the same bin;
//     survivors above it join the winners, the others leave.  The rounds stop when winners plus survivors are exactly
//     k (set output) or fit one ranking (sorted output).  A CTA whose survivors overflow
//     its shared memory rescans its slice (in L2) each round instead.
//  4. Output: the set -- each CTA writes its lists at offsets given by a prefix over the
//     CTAs' published counts (winners of all CTAs first, then survivors; a fixed order);
//     or sorted -- every CTA copies its lists into CTA 0, which ranks them.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int TK_T = 1024;           // threads per CTA
constexpr int TK_BINS = kHistBins;   // 2048: widest digit
constexpr int TK_KMAX = 2048;        // largest k; winners capacity per CTA
constexpr int TK_SCAP = 16384;       // survivors held in shared memory per CTA
constexpr int TK_MAXCL = 16;         // cluster size limit (non-portable above 8)
constexpr int TK_SLICE = 16384;      // scores per CTA the cluster size is chosen for

struct TopkArgs {
    const float* scores;
    int B;
    int nq;  // decode mode: query positions per request
    int64_t G;
    const int64_t* offsets;
    const int64_t* n_tokens;
    int ratio;
    int64_t score_stride;
    int k;
    int32_t* idx_out;
    uint32_t* keys_out;
    int sorted;              // 1: output ordered by (score desc, index asc); 0: the set, in a fixed order
    int hist_fused;          // digit 0's histogram (block words [0, kHistBins)) comes from the score kernel
    uint32_t* hist;          // [B][kHistBlock], zeroed before the launch: one histogram per digit
    int32_t* status;
};

struct TkSmem {
    uint32_t hist[2][TK_BINS];  // this CTA's counts of the round's digit (read by the whole cluster)
    uint32_t okey[TK_KMAX];     // this CTA's winners (CTA 0, sorted output: the cluster's union)
    int32_t oidx[TK_KMAX];
    uint32_t ckey[TK_SCAP];     // this CTA's survivors
    int32_t cidx[TK_SCAP];
    uint64_t sortbuf[TK_KMAX];
    uint32_t wsum[32];
    uint32_t pub[2];            // published {winners, survivors} of this CTA
    uint32_t pw, ps, W, Cs;     // output offsets of this CTA's lists and the cluster's totals
    int n_sel, n_cand, n_new, over;
    uint32_t bin, above, cnt;
};

__device__ __forceinline__ void request_span(const TopkArgs& a, int b, const float*& sc, int64_t& G) {
    if (a.offsets) {
        const int64_t o0 = a.offsets[b], o1 = a.offsets[b + 1];
        sc = a.scores + o0;
        G = o1 - o0;
    } else if (a.n_tokens) {
        sc = a.scores + (int64_t)b * a.score_stride;
        G = query_tokens(a.n_tokens, b, a.nq) / a.ratio;
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

// prefix match of (key, index) on digits 0 .. d-1
__device__ __forceinline__ bool prefix_match(const uint32_t (&bins)[6], int d, uint32_t key, int32_t idx) {
    if ((key >> 21) != bins[0]) return false;
    for (int e = 1; e < d; ++e)
        if (digit_of(e, key, idx) != bins[e]) return false;
    return true;
}

// Block-wide exclusive offsets for this thread's ns winners and nc survivors (each < 2^16
// per block), appended after the current lists; updates the counters.  Every thread calls it.
__device__ __forceinline__ void ordered_reserve(TkSmem& sm, uint32_t ns, uint32_t nc, int& bs, int& bc) {
    uint32_t tot;
    const uint32_t ex = block_scan(sm, (ns << 16) | nc, &tot);
    bs = sm.n_sel + (int)(ex >> 16);
    bc = sm.n_cand + (int)(ex & 0xFFFFu);
    __syncthreads();  // every thread has read the counters
    if (threadIdx.x == 0) {
        sm.n_sel += (int)(tot >> 16);
        sm.n_cand += (int)(tot & 0xFFFFu);
    }
    __syncthreads();
}

// The round's histogram of the whole request, summed over the cluster's CTAs through
// distributed shared memory: after one cluster barrier (release/acquire: every CTA's counts
// in its own hist[hb] are complete and visible), thread t reads its two bins from every CTA's
// shared memory, and every CTA finds the same bin of `need`.  hist[hb] is not written again
// before the next round's barrier (the rounds alternate between two histograms), so no CTA
// overwrites counts another may still be reading.
__device__ __forceinline__ void cluster_find_bin(TkSmem& sm, int hb, int nbins, uint32_t need) {
    cluster_sync();
    const int cl = (int)gridDim.x;
    const int bh = nbins - 1 - 2 * (int)threadIdx.x, bl = bh - 1;
    uint32_t th = 0, tl = 0;
    if (bl >= 0) {
        const uint32_t ah = smem_u32(&sm.hist[hb][bh]), al = smem_u32(&sm.hist[hb][bl]);
        uint32_t vh[TK_MAXCL], vl[TK_MAXCL];
#pragma unroll
        for (int r = 0; r < TK_MAXCL; ++r) {  // all loads in flight, then the sums
            vh[r] = r < cl ? ld_dsmem_u32(mapa(ah, (uint32_t)r)) : 0u;
            vl[r] = r < cl ? ld_dsmem_u32(mapa(al, (uint32_t)r)) : 0u;
        }
#pragma unroll
        for (int r = 0; r < TK_MAXCL; ++r) {
            th += vh[r];
            tl += vl[r];
        }
    }
    find_bin_vals(sm, th, tl, nbins, need);
}

__global__ void __launch_bounds__(TK_T, 1) topk_cluster_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    const int tid = threadIdx.x;
    pdl_wait();               // scores (and the fused histogram) come from the preceding kernel
    pdl_launch_dependents();
    const int cl = (int)gridDim.x;  // one cluster per request
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.y;
    const float* sc;
    int64_t G;
    request_span(a, b, sc, G);
    const int k = a.k;
    int32_t* out = a.idx_out + (int64_t)b * k;
    uint32_t* kout = a.keys_out ? a.keys_out + (int64_t)b * k : nullptr;
    const bool all_in = G <= k;  // every candidate is selected
    const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15) == 0;
    const int64_t slice = (((G + cl - 1) / cl) + 3) & ~int64_t(3);
    const int64_t lo = min((int64_t)rank * slice, G), hi = min(lo + slice, G);
    for (int i = tid; i < 2 * TK_BINS; i += TK_T) (&sm.hist[0][0])[i] = 0;
    if (tid == 0) {
        sm.n_sel = 0;
        sm.n_cand = 0;
        sm.over = 0;
    }
    __syncthreads();

    // ---- 1. first digit
    uint32_t bins[6] = {0, 0, 0, 0, 0, 0};
    uint32_t need = (uint32_t)k, tot_w = (uint32_t)(G < k ? G : k), tot_c = 0;
    if (!all_in) {
        if (a.hist_fused) {
            find_bin_global(sm, a.hist + (int64_t)b * kHistBlock, TK_BINS, need);
        } else {
            for (int64_t base = lo; base < hi; base += 4 * TK_T) {  // the same trip count for every thread
                uint32_t key[4];
                const int64_t pos = base + 4 * tid;
                load4(sc, pos, hi, vec, key);
#pragma unroll
                for (int q = 0; q < 4; ++q) hist_add(sm.hist[0], key[q] >> 21, pos + q < hi);
            }
            cluster_find_bin(sm, 0, TK_BINS, need);
        }
        bins[0] = sm.bin;
        need -= sm.above;
        tot_w = sm.above;
        tot_c = sm.cnt;
    }
    // ---- 2. one scan of the slice: winners (first digit above b0, or all) and survivors.
    //      Passes of TK_T * 16 scores: all 16 of a thread in flight, one reservation per pass.
    for (int64_t base = lo; base < hi; base += (int64_t)16 * TK_T) {
        uint32_t key[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t k4[4];
            load4(sc, base + 4 * ((int64_t)tid + (int64_t)j * TK_T), hi, vec, k4);
#pragma unroll
            for (int q = 0; q < 4; ++q) key[4 * j + q] = k4[q];
        }
        uint32_t ns = 0, nc = 0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int64_t p = base + 4 * ((int64_t)tid + (int64_t)(e >> 2) * TK_T) + (e & 3);
            const bool in = p < hi;
            const uint32_t d = key[e] >> 21;
            ns += (in && (all_in || d > bins[0])) ? 1u : 0u;
            nc += (in && !all_in && d == bins[0]) ? 1u : 0u;
        }
        // element order within a pass: 4-score group j of every thread, by thread -- index
        // order within each group column, so each list is sorted by index within a pass
        // column; the lists only need a fixed order
        int bs, bc;
        ordered_reserve(sm, ns, nc, bs, bc);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int64_t p = base + 4 * ((int64_t)tid + (int64_t)(e >> 2) * TK_T) + (e & 3);
            const bool in = p < hi;
            const uint32_t d = key[e] >> 21;
            if (in && (all_in || d > bins[0])) {
                if (bs < TK_KMAX) { sm.okey[bs] = key[e]; sm.oidx[bs] = (int32_t)p; }
                else raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                ++bs;
            } else if (in && !all_in && d == bins[0]) {
                if (bc < TK_SCAP) { sm.ckey[bc] = key[e]; sm.cidx[bc] = (int32_t)p; }
                ++bc;
            }
        }
    }
    bool implicit = sm.n_cand > TK_SCAP;  // this CTA's survivors did not fit: rounds rescan the slice

    // ---- 3. rounds over the next digits
    const int target = a.sorted ? (k <= 1024 ? 1024 : TK_KMAX) : k;
    for (int d = 1; d <= 5 && (int)(tot_w + tot_c) > target; ++d) {
        const int hb = d & 1, nb = digit_bins(d);
        for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[hb][i] = 0;
        __syncthreads();
        if (!implicit) {
            const int n = sm.n_cand;
            for (int i0 = 0; i0 < n; i0 += TK_T) {
                const int i = i0 + tid;
                const bool in = i < n;
                hist_add(sm.hist[hb], in ? digit_of(d, sm.ckey[i], sm.cidx[i]) : 0u, in);
            }
        } else {
            for (int64_t base = lo; base < hi; base += 4 * TK_T) {
                uint32_t key[4];
                const int64_t pos = base + 4 * tid;
                load4(sc, pos, hi, vec, key);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < hi && prefix_match(bins, d, key[q], idx);
                    hist_add(sm.hist[hb], in ? digit_of(d, key[q], idx) : 0u, in);
                }
            }
        }
        cluster_find_bin(sm, hb, nb, need);
        const uint32_t dbin = sm.bin;
        need -= sm.above;
        tot_w += sm.above;
        tot_c = sm.cnt;
        bins[d] = dbin;
        if (!implicit) {
            // in-place, order-preserving: a chunk is read by everyone before any of it is rewritten
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
            if (tid == 0) sm.n_cand = 0;
            __syncthreads();
            for (int64_t base = lo; base < hi; base += 4 * TK_T) {
                uint32_t key[4];
                const int64_t pos = base + 4 * tid;
                load4(sc, pos, hi, vec, key);
                uint32_t ns = 0, nc = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < hi && prefix_match(bins, d, key[q], idx);
                    const uint32_t dv = digit_of(d, key[q], idx);
                    ns += (in && dv > dbin) ? 1u : 0u;
                    nc += (in && dv == dbin) ? 1u : 0u;
                }
                int bs, bc;
                ordered_reserve(sm, ns, nc, bs, bc);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < hi && prefix_match(bins, d, key[q], idx);
                    const uint32_t dv = digit_of(d, key[q], idx);
                    if (in && dv > dbin) {
                        if (bs < TK_KMAX) { sm.okey[bs] = key[q]; sm.oidx[bs] = idx; }
                        ++bs;
                    } else if (in && dv == dbin) {
                        if (bc < TK_SCAP) { sm.ckey[bc] = key[q]; sm.cidx[bc] = idx; }
                        ++bc;
                    }
                }
            }
            implicit = sm.n_cand > TK_SCAP;
        }
        __syncthreads();
    }

    // ---- 4. output: offsets of this CTA's lists from the cluster's published counts
    const int my_w = min(sm.n_sel, TK_KMAX), my_c = implicit ? 0 : min(sm.n_cand, TK_SCAP);
    if (tid == 0) {
        sm.pub[0] = (uint32_t)my_w;
        sm.pub[1] = (uint32_t)my_c;
        if (implicit) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);  // (cannot happen: the rounds end exact)
    }
    cluster_sync();
    if (tid < 32) {  // lane c reads CTA c's counts; exclusive prefix below this CTA and the totals
        const int lane = tid;
        const uint32_t w = lane < cl ? ld_dsmem_u32(mapa(smem_u32(&sm.pub[0]), (uint32_t)lane)) : 0u;
        const uint32_t sv = lane < cl ? ld_dsmem_u32(mapa(smem_u32(&sm.pub[1]), (uint32_t)lane)) : 0u;
        uint32_t xw = w, xs = sv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yw = __shfl_up_sync(0xffffffffu, xw, o), ys = __shfl_up_sync(0xffffffffu, xs, o);
            if (lane >= o) { xw += yw; xs += ys; }
        }
        if (lane == (int)rank) {
            sm.pw = xw - w;
            sm.ps = xs - sv;
        }
        if (lane == 31) {
            sm.W = xw;
            sm.Cs = xs;
        }
    }
    __syncthreads();
    const uint32_t pw = sm.pw, ps = sm.ps, W = sm.W, Cs = sm.Cs;
    if (!a.sorted) {
        for (int i = tid; i < my_w; i += TK_T) {
            const uint32_t o = pw + (uint32_t)i;
            if (o < (uint32_t)k) {
                out[o] = sm.oidx[i];
                if (kout) kout[o] = sm.okey[i];
            }
        }
        for (int i = tid; i < my_c; i += TK_T) {
            const uint32_t o = W + ps + (uint32_t)i;
            if (o < (uint32_t)k) {
                out[o] = sm.cidx[i];
                if (kout) kout[o] = sm.ckey[i];
            }
        }
        if (rank == 0)
            for (int i = (int)(W + Cs) + tid; i < k; i += TK_T) {
                out[i] = -1;
                if (kout) kout[i] = 0u;
            }
        cluster_sync();  // the counts stay readable until every CTA has read them
        return;
    }
    // sorted: every CTA copies its lists into CTA 0 (winners of all CTAs, then survivors)
    const uint32_t okey0 = mapa(smem_u32(&sm.okey[0]), 0u), oidx0 = mapa(smem_u32(&sm.oidx[0]), 0u);
    if (rank != 0)
        for (int i = tid; i < my_w; i += TK_T) {
            const uint32_t o = pw + (uint32_t)i;
            if (o < (uint32_t)TK_KMAX) {
                st_dsmem_u32(okey0 + 4u * o, sm.okey[i]);
                st_dsmem_u32(oidx0 + 4u * o, (uint32_t)sm.oidx[i]);
            }
        }
    for (int i = tid; i < my_c; i += TK_T) {
        const uint32_t o = W + ps + (uint32_t)i;
        if (o < (uint32_t)TK_KMAX) {
            st_dsmem_u32(okey0 + 4u * o, sm.ckey[i]);
            st_dsmem_u32(oidx0 + 4u * o, (uint32_t)sm.cidx[i]);
        }
    }
    cluster_sync();  // CTA 0 holds the union
    if (rank != 0) return;
    rank_scatter(sm, (int)min(W + Cs, (uint32_t)TK_KMAX), k, out, kout);
}

// ------------------------------------------------------------------ host side
constexpr int kTopkMaxDevices = 64;
static int g_max_cluster[kTopkMaxDevices];  // largest schedulable cluster of the kernel, per device
static std::mutex g_topk_mu;

// CTAs per request: about TK_SLICE scores each, a power of two, at most `max_cl`.
static int topk_cluster_size(int64_t max_G, int max_cl) {
    int c = 1;
    while ((int64_t)c * TK_SLICE < max_G && c < TK_MAXCL) c <<= 1;
    while (c > max_cl && c > 1) c >>= 1;
    return c;
}

size_t topk_lists_bytes(int B, int64_t max_G, int k) {
    (void)B;
    (void)max_G;
    (void)k;
    return 0;  // the lists live in the cluster's shared memory
}

cudaError_t launch_topk(const TopkLaunch& h, cudaStream_t s, bool pdl) {
    TopkArgs a;
    a.scores = h.scores;
    a.B = h.B;
    a.G = h.G;
    a.offsets = h.offsets;
    a.n_tokens = h.n_tokens;
    a.nq = h.nq > 1 ? h.nq : 1;
    a.ratio = h.ratio;
    a.score_stride = h.score_stride;
    a.k = h.k;
    a.idx_out = h.idx_out;
    a.keys_out = h.keys_out;
    a.sorted = h.sorted ? 1 : 0;
    a.hist_fused = h.hist_fused ? 1 : 0;
    a.hist = h.hist;
    a.status = h.status;
    const size_t smem = sizeof(TkSmem);
    cudaError_t e = set_func_attr_once((const void*)topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
    if (e == cudaSuccess)
        e = set_func_attr_once((const void*)topk_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kTopkMaxDevices) return cudaErrorInvalidDevice;
    int max_cl;
    {
        std::lock_guard<std::mutex> lk(g_topk_mu);
        if (!g_max_cluster[dev]) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(TK_MAXCL, 1, 1);
            q.blockDim = dim3(TK_T, 1, 1);
            q.dynamicSmemBytes = smem;
            int mc = 0;
            if (cudaOccupancyMaxPotentialClusterSize(&mc, topk_cluster_kernel, &q) != cudaSuccess || mc < 1) {
                cudaGetLastError();
                mc = 8;  // portable cluster size
            }
            g_max_cluster[dev] = mc < TK_MAXCL ? mc : TK_MAXCL;
        }
        max_cl = g_max_cluster[dev];
    }
    const int cl = topk_cluster_size(h.max_G, max_cl);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    cfg.gridDim = dim3((unsigned)cl, (unsigned)h.B, 1);
    cfg.blockDim = dim3(TK_T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, a);
}

}  // namespace csa
