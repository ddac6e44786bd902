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
constexpr int TK_SCAP = 16384;       // survivors list capacity (global and shared)
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
    uint32_t* hist;   // [B][kHistBlock]: first-digit histogram, then the control words
    uint2* wlist;     // [B][TK_KMAX] winners {key, index}
    uint2* slist;     // [B][TK_SCAP] survivors
    int32_t* status;
};

struct TkSmem {
    uint32_t hist[TK_BINS];
    uint32_t okey[TK_KMAX];     // winners, then the union to sort
    int32_t oidx[TK_KMAX];
    uint32_t ckey[TK_SCAP];     // survivors
    int32_t cidx[TK_SCAP];
    uint64_t sortbuf[2][1024];
    uint32_t wsum[32];
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

__device__ __forceinline__ int warp_alloc(int* counter, bool pred) {
    const unsigned m = __ballot_sync(0xffffffffu, pred);
    if (m == 0) return -1;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(m) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(m));
    base = __shfl_sync(0xffffffffu, base, leader);
    return pred ? base + __popc(m & ((1u << lane) - 1u)) : -1;
}

// Slots for this thread's ns winners and nc survivors (each < 2^16 per warp): one atomic
// per non-empty list per warp.
__device__ __forceinline__ void warp_reserve(int* cs, int* cc, uint32_t ns, uint32_t nc, int& bs, int& bc) {
    const int lane = threadIdx.x & 31;
    const uint32_t v = (ns << 16) | nc;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, x, 31);
    int b_s = 0, b_c = 0;
    if (lane == 31) {
        if (tot >> 16) b_s = atomicAdd(cs, (int)(tot >> 16));
        if (tot & 0xFFFFu) b_c = atomicAdd(cc, (int)(tot & 0xFFFFu));
    }
    b_s = __shfl_sync(0xffffffffu, b_s, 31);
    b_c = __shfl_sync(0xffffffffu, b_c, 31);
    const uint32_t ex = x - v;
    bs = b_s + (int)(ex >> 16);
    bc = b_c + (int)(ex & 0xFFFFu);
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

enum { HIST_GLOBAL = 0, HIST_LOCAL = 1 };

// The bin holding the need-th largest element counted from the top bin, from a
// global histogram (written by an earlier kernel) or this CTA's sm.hist.  Writes
// sm.bin, sm.above (count in higher bins) and sm.cnt (count in the bin).
__device__ __forceinline__ void find_bin(TkSmem& sm, int mode, const uint32_t* ghist, int nbins, uint32_t need) {
    const int t = threadIdx.x;
    const int bh = nbins - 1 - 2 * t, bl = nbins - 2 - 2 * t;  // this thread's two bins, high first
    uint32_t th = 0, tl = 0;
    if (bl >= 0) {
        if (mode == HIST_GLOBAL) {
            th = __ldg(ghist + bh);
            tl = __ldg(ghist + bl);
        } else {
            th = sm.hist[bh];
            tl = sm.hist[bl];
        }
    }
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

__device__ __forceinline__ bool kv_greater(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Sort okey/oidx[0..total) by (key desc, index asc) and write k outputs (-1 padding).
__device__ void sort_and_write(TkSmem& sm, uint32_t total, int k, int32_t* out, uint32_t* kout) {
    const int tid = threadIdx.x, lane = tid & 31;
    if (total > (uint32_t)TK_KMAX) total = TK_KMAX;
    int n2 = 1;
    while (n2 < (int)total) n2 <<= 1;
    if (n2 <= 1024) {
        // one element per thread of the first max(n2, 32) threads; composite = key << 32 |
        // (0x7FFFFFFF - idx) so that larger is better.  Strides below a warp use shuffles,
        // larger ones exchange through shared memory behind a barrier of just these warps.
        const int nt = n2 < 32 ? 32 : n2;
        uint64_t v = 0;
        if (tid < nt) {
            if (tid < (int)total) v = ((uint64_t)sm.okey[tid] << 32) | (uint32_t)(0x7FFFFFFF - sm.oidx[tid]);
            int buf = 0;
            for (int size = 2; size <= n2; size <<= 1) {
                for (int j = size >> 1; j > 0; j >>= 1) {
                    uint64_t pv;
                    if (j >= 32) {
                        sm.sortbuf[buf][tid] = v;
                        asm volatile("bar.sync 2, %0;" ::"r"(nt) : "memory");
                        pv = sm.sortbuf[buf][tid ^ j];
                        buf ^= 1;
                    } else {
                        pv = __shfl_xor_sync(0xffffffffu, v, j);
                    }
                    const bool up = (tid & size) == 0, lower = (tid & j) == 0;
                    const uint64_t mx = v > pv ? v : pv, mn = v > pv ? pv : v;
                    v = (up == lower) ? mx : mn;
                }
            }
        }
        if (tid < k) {
            const bool ok = tid < (int)total;
            out[tid] = ok ? (int32_t)(0x7FFFFFFF - (uint32_t)v) : -1;
            if (kout) kout[tid] = ok ? (uint32_t)(v >> 32) : 0u;
        }
        for (int i = tid + TK_T; i < k; i += TK_T) {
            out[i] = -1;
            if (kout) kout[i] = 0u;
        }
        return;
    }
    // n2 = 2048: shared-memory bitonic network
    for (int i = (int)total + tid; i < n2; i += TK_T) {
        sm.okey[i] = 0u;
        sm.oidx[i] = 0x7FFFFFFF;
    }
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = tid; i < n2; i += TK_T) {
                const int j = i ^ stride;
                if (j > i) {
                    const uint32_t ki = sm.okey[i], kj = sm.okey[j];
                    const int32_t ii = sm.oidx[i], ij = sm.oidx[j];
                    const bool first_half = (i & size) == 0;
                    const bool swap = first_half ? kv_greater(kj, ij, ki, ii) : kv_greater(ki, ii, kj, ij);
                    if (swap) {
                        sm.okey[i] = kj; sm.oidx[i] = ij;
                        sm.okey[j] = ki; sm.oidx[j] = ii;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = tid; i < k; i += TK_T) {
        const bool ok = i < (int)total;
        out[i] = ok ? sm.oidx[i] : -1;
        if (kout) kout[i] = ok ? sm.okey[i] : 0u;
    }
    (void)lane;
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

__global__ void __launch_bounds__(TK_T, 1) topk_select_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    const int tid = threadIdx.x;
    pdl_wait();               // scores (and the fused histogram) come from the preceding kernel
    pdl_launch_dependents();
    const int b = blockIdx.y;
    const float* sc;
    int64_t G;
    request_span(a, b, sc, G);
    const int k = a.k;
    uint32_t* ghist = a.hist + (int64_t)b * kHistBlock;
    uint32_t* ctl = ghist + kHistBins;  // [0] winners, [1] survivors, [2] finished CTAs
    uint2* wl = a.wlist + (int64_t)b * TK_KMAX;
    uint2* sl = a.slist + (int64_t)b * TK_SCAP;
    int32_t* out = a.idx_out + (int64_t)b * k;
    uint32_t* kout = a.keys_out ? a.keys_out + (int64_t)b * k : nullptr;
    const bool all_in = G <= k;  // every candidate is selected
    const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15) == 0;

    // ---- A. first digit from the request's histogram; one scan of this CTA's slice
    uint32_t b0 = 0;
    if (!all_in) {
        find_bin(sm, HIST_GLOBAL, ghist, TK_BINS, (uint32_t)k);
        b0 = sm.bin;
    }
    const int64_t chunk = (((G + gridDim.x - 1) / gridDim.x) + 3) & ~int64_t(3);
    const int64_t lo = min((int64_t)blockIdx.x * chunk, G), hi = min(lo + chunk, G);
    for (int64_t base = lo; base < hi; base += TK_CHUNK) {
        const int64_t pos = base + 4 * tid;
        uint32_t key[4];
        load4(sc, pos, hi, vec, key);
        uint32_t ns = 0, nc = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = pos + q < hi;
            const uint32_t d = key[q] >> 21;
            ns += (in && (all_in || d > b0)) ? 1u : 0u;
            nc += (in && !all_in && d == b0) ? 1u : 0u;
        }
        if (!__any_sync(0xffffffffu, (ns | nc) != 0)) continue;
        int bs, bc;
        warp_reserve(reinterpret_cast<int*>(&ctl[0]), reinterpret_cast<int*>(&ctl[1]), ns, nc, bs, bc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = pos + q < hi;
            const uint32_t d = key[q] >> 21;
            if (in && (all_in || d > b0)) {
                if (bs < TK_KMAX) wl[bs] = make_uint2(key[q], (uint32_t)(pos + q));
                else raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                ++bs;
            } else if (in && !all_in && d == b0) {
                if (bc < TK_SCAP) sl[bc] = make_uint2(key[q], (uint32_t)(pos + q));
                ++bc;
            }
        }
    }
    // ---- the last CTA of the request to finish goes on
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        sm.last = atomicAdd(&ctl[2], 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    // ---- B. refine the survivors
    if (tid == 0) {
        const uint32_t nw = __ldcg(&ctl[0]);
        sm.n_sel = (int)min(nw, (uint32_t)TK_KMAX);
        sm.n_cand = (int)__ldcg(&ctl[1]);
    }
    __syncthreads();
    const int n_w0 = sm.n_sel;
    bool implicit = sm.n_cand > TK_SCAP;  // survivors list incomplete: the digits run over the scores
    for (int i = tid; i < n_w0; i += TK_T) {
        const uint2 v = __ldcg(wl + i);
        sm.okey[i] = v.x;
        sm.oidx[i] = (int32_t)v.y;
    }
    if (!implicit)
        for (int i = tid; i < sm.n_cand; i += TK_T) {
            const uint2 v = __ldcg(sl + i);
            sm.ckey[i] = v.x;
            sm.cidx[i] = (int32_t)v.y;
        }
    __syncthreads();
    uint32_t need = all_in ? 0u : (uint32_t)k - (uint32_t)n_w0;
    const int sort_max = k <= 1024 ? 1024 : TK_KMAX;
    uint32_t bins[6] = {b0, 0, 0, 0, 0, 0};
    // prefix match of (key, index) on digits 0 .. d-1 (implicit mode)
    auto matches = [&](int d, uint32_t key, int32_t idx) {
        if ((key >> 21) != bins[0]) return false;
        for (int e = 1; e < d; ++e)
            if (digit_of(e, key, idx) != bins[e]) return false;
        return true;
    };
    for (int d = 1; d <= 5 && sm.n_sel + sm.n_cand > sort_max; ++d) {
        const int nb = digit_bins(d);
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
                uint32_t key[4];
                const int64_t pos = p0 + 4 * tid;
                load4(sc, pos, G, vec, key);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < G && matches(d, key[q], idx);
                    hist_add(sm.hist, in ? digit_of(d, key[q], idx) : 0u, in);
                }
            }
        }
        __syncthreads();
        find_bin(sm, HIST_LOCAL, nullptr, nb, need);
        const uint32_t bin = sm.bin, n_bin = sm.cnt;
        need -= sm.above;
        bins[d] = bin;
        if (!implicit) {
            // in-place compaction: a chunk is read by everyone before any of it is overwritten
            const int n = sm.n_cand;
            if (tid == 0) sm.n_new = 0;
            __syncthreads();
            for (int i0 = 0; i0 < n; i0 += TK_T) {
                const int i = i0 + tid;
                const bool in = i < n;
                const uint32_t key = in ? sm.ckey[i] : 0u;
                const int32_t idx = in ? sm.cidx[i] : 0;
                __syncthreads();
                const uint32_t dv = digit_of(d, key, idx);
                const int so = warp_alloc(&sm.n_sel, in && dv > bin);
                if (so >= 0 && so < TK_KMAX) { sm.okey[so] = key; sm.oidx[so] = idx; }
                const int c = warp_alloc(&sm.n_new, in && dv == bin);
                if (c >= 0) { sm.ckey[c] = key; sm.cidx[c] = idx; }
            }
            __syncthreads();
            if (tid == 0) sm.n_cand = sm.n_new;
        } else {
            const bool gather = n_bin <= (uint32_t)TK_SCAP;
            if (tid == 0) sm.n_cand = 0;
            __syncthreads();
            for (int64_t p0 = 0; p0 < G; p0 += 4 * TK_T) {
                uint32_t key[4];
                const int64_t pos = p0 + 4 * tid;
                load4(sc, pos, G, vec, key);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int32_t idx = (int32_t)(pos + q);
                    const bool in = pos + q < G && matches(d, key[q], idx);
                    const uint32_t dv = digit_of(d, key[q], idx);
                    const int so = warp_alloc(&sm.n_sel, in && dv > bin);
                    if (so >= 0 && so < TK_KMAX) { sm.okey[so] = key[q]; sm.oidx[so] = idx; }
                    const int c = warp_alloc(&sm.n_cand, gather && in && dv == bin);
                    if (c >= 0 && c < TK_SCAP) { sm.ckey[c] = key[q]; sm.cidx[c] = idx; }
                }
            }
            __syncthreads();
            if (tid == 0 && !gather) sm.n_cand = (int)n_bin;
            implicit = !gather;
        }
        __syncthreads();
    }
    // ---- the union of winners and survivors fits one sort
    const int n_w = sm.n_sel, n_c = implicit ? 0 : sm.n_cand;
    if (tid == 0 && n_w + n_c > TK_KMAX) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    for (int i = tid; i < n_c && n_w + i < TK_KMAX; i += TK_T) {
        sm.okey[n_w + i] = sm.ckey[i];
        sm.oidx[n_w + i] = sm.cidx[i];
    }
    __syncthreads();
    sort_and_write(sm, (uint32_t)min(n_w + n_c, TK_KMAX), k, out, kout);
}

static int g_sms = 0;
static int sm_count() {
    if (!g_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev);
    }
    return g_sms;
}

static TopkArgs topk_args(const TopkLaunch& h) {
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
    a.hist = h.hist;
    a.wlist = reinterpret_cast<uint2*>(h.lists);
    a.slist = reinterpret_cast<uint2*>(h.lists) + (size_t)h.B * TK_KMAX;
    a.status = h.status;
    return a;
}

size_t topk_lists_bytes(int B) { return (size_t)B * (TK_KMAX + TK_SCAP) * sizeof(uint2); }

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
    // slices of about TK_CHUNK scores, at most one wave of CTAs over the batch
    int64_t per = (h.max_G + TK_CHUNK - 1) / TK_CHUNK;
    const int64_t cap = (sm_count() + h.B - 1) / h.B;
    if (per > cap) per = cap;
    if (per < 1) per = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((unsigned)per, (unsigned)h.B, 1);
    cfg.blockDim = dim3(TK_T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, topk_select_kernel, a);
}

}  // namespace csa
