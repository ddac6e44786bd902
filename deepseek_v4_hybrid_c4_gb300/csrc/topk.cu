// Stage 3: exact top-k of the index scores by cluster radix select (the pages'
// "Lightning TopK": per-CTA histograms over N/8 candidates reduced inside a
// cluster of 8 to a threshold tau, then a local scatter of the entries above
// tau -- "SGLang 如何为 DeepSeek V4 打造「Day-0」推理加速", sec. "创新 2";
// "DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "Kernel 層一堆狠活").
//
// Order: descending order-preserving 32-bit key of the fp32 score, ties to the
// lower index (a total order, so the selected set and its order are unique).
//
// One cluster of 8 CTAs per request; CTA r owns the contiguous index slice
// [r*S, r*S+S).  Digits of the key: bits 31..21, 20..10, 9..0.
//  1. First digit: its histogram over the whole request -- ready-made by the
//     score kernel in the fused decode step, otherwise built per CTA and summed
//     across the cluster through distributed shared memory -- gives the bin b0
//     holding the k-th key.
//  2. Each CTA scans its slice once (16 scores in flight per thread): keys in
//     higher bins are winners, keys in b0 are survivors.
//  3. Fast path (the survivors of all 8 CTAs fit CTA 0's gather buffer): every
//     CTA copies its winners and survivors into CTA 0 through DSMEM and CTA 0
//     finishes alone -- two more digits over the survivors, then the lowest-index
//     ties at the exact threshold -- with no further cluster barrier.
//     Otherwise every CTA keeps refining its survivors with cluster-reduced
//     histograms (re-reading L2 when more than CAP survive) and the ties are
//     taken lowest index first across the index-ordered slices.
//  4. CTA 0 sorts the k winners by (key desc, index asc) with a bitonic network
//     kept in registers (shuffles) except for strides of a warp or more.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int TK_CL = 8;
constexpr int TK_T = 1024;
constexpr int TK_BINS = kHistBins;   // 2048: widest digit
constexpr int TK_CAP = 10240;        // survivors kept per CTA
constexpr int TK_KMAX = 2048;
constexpr int TK_GCAP = 6144;        // survivors CTA 0 can take from the whole cluster
constexpr int TK_V = 16;             // scores per thread per scan iteration

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
    const uint32_t* hist;
    int32_t* status;
};

struct TkSmem {
    uint32_t hist[2][TK_BINS];
    uint32_t ckey[TK_CAP];      // this CTA's survivors
    int32_t cidx[TK_CAP];
    uint32_t skey[TK_KMAX];     // this CTA's winners
    int32_t sidx[TK_KMAX];
    uint32_t okey[TK_KMAX];     // CTA 0: the cluster's winners
    int32_t oidx[TK_KMAX];
    uint32_t gkey[TK_GCAP];     // CTA 0: the cluster's survivors (fast path)
    int32_t gidx[TK_GCAP];
    uint64_t sortbuf[2][1024];
    uint32_t xchg[8];
    uint32_t wsum[32];
    int n_cand, n_sel, n_new, overflow, n_out;
    uint32_t bin, above, cnt, taken;
};

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

// Slots for this thread's ns winners and nc survivors: one atomic per list per warp.
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
        b_s = atomicAdd(cs, (int)(tot >> 16));
        b_c = atomicAdd(cc, (int)(tot & 0xFFFFu));
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

enum { HIST_GLOBAL = 0, HIST_CLUSTER = 1, HIST_LOCAL = 2 };

// The bin holding the need-th largest key counted from the top bin, from the
// global histogram, the sum of the 8 CTAs' histograms (DSMEM) or this CTA's own.
// Writes sm.bin and sm.above (count in higher bins).
__device__ __forceinline__ void find_bin(TkSmem& sm, int mode, const uint32_t* ghist, int hb, int nbins,
                                         uint32_t need) {
    const int t = threadIdx.x;
    const int bh = nbins - 1 - 2 * t, bl = nbins - 2 - 2 * t;  // this thread's two bins, high first
    uint32_t th = 0, tl = 0;
    if (bl >= 0) {
        if (mode == HIST_GLOBAL) {
            th = __ldg(ghist + bh);
            tl = __ldg(ghist + bl);
        } else if (mode == HIST_LOCAL) {
            th = sm.hist[hb][bh];
            tl = sm.hist[hb][bl];
        } else {
            const uint32_t ah = smem_u32(&sm.hist[hb][bh]), al = smem_u32(&sm.hist[hb][bl]);
            uint32_t vh[TK_CL], vl[TK_CL];
#pragma unroll
            for (int c = 0; c < TK_CL; ++c) {
                vh[c] = ld_dsmem_u32(mapa(ah, c));
                vl[c] = ld_dsmem_u32(mapa(al, c));
            }
#pragma unroll
            for (int c = 0; c < TK_CL; ++c) {
                th += vh[c];
                tl += vl[c];
            }
        }
    }
    uint32_t total;
    const uint32_t excl = block_scan(sm, th + tl, &total);
    if (bl >= 0) {
        if (th > 0 && excl < need && need <= excl + th) {
            sm.bin = (uint32_t)bh;
            sm.above = excl;
        } else if (tl > 0 && excl + th < need && need <= excl + th + tl) {
            sm.bin = (uint32_t)bl;
            sm.above = excl + th;
        }
    }
    __syncthreads();
}

// Keys of TK_V scores of the slice for this thread: element j*4+q is index
// base + 4*(tid + (j/1)*TK_T) + q (coalesced float4 loads when the slice is 16-byte aligned).
__device__ __forceinline__ void load_keys(const float* sc, int64_t base, int64_t hi, bool vec, uint32_t (&key)[TK_V],
                                          int64_t (&pos)[TK_V / 4]) {
    const int tid = threadIdx.x;
#pragma unroll
    for (int j = 0; j < TK_V / 4; ++j) {
        pos[j] = base + 4 * ((int64_t)tid + (int64_t)j * TK_T);
        float v[4];
        if (vec && pos[j] + 3 < hi) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(sc + pos[j]));
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) v[q] = pos[j] + q < hi ? __ldg(sc + pos[j] + q) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) key[j * 4 + q] = score_key(v[q]);
    }
}

__device__ __forceinline__ bool kv_greater(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// CTA 0: sort okey/oidx[0..total) by (key desc, index asc), write k outputs (-1 padding).
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

__global__ void __launch_bounds__(TK_T, 1) topk_kernel(TopkArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    TkSmem& sm = *reinterpret_cast<TkSmem*>(tk_raw);
    const int tid = threadIdx.x;
    pdl_wait();               // scores (and the fused histogram) come from the preceding kernel
    pdl_launch_dependents();
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / TK_CL;

    const float* sc;
    int64_t G;
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
    const int k = a.k;
    const int64_t slice = ((G + TK_CL - 1) / TK_CL + 3) & ~int64_t(3);
    const int64_t lo = min((int64_t)rank * slice, G), hi = min(lo + slice, G);
    const bool vec = (reinterpret_cast<uintptr_t>(sc + lo) & 15) == 0;
    int32_t* out = a.idx_out + (int64_t)b * k;
    uint32_t* kout = a.keys_out ? a.keys_out + (int64_t)b * k : nullptr;

    if (tid == 0) {
        sm.n_cand = 0;
        sm.n_sel = 0;
        sm.overflow = 0;
        sm.n_out = 0;
    }
    __syncthreads();

    if (G > k) {
        uint32_t need = (uint32_t)k;
        // ---- 1. first digit (bits 31..21)
        if (a.hist) {
            find_bin(sm, HIST_GLOBAL, a.hist + (int64_t)b * kHistBins, 0, 2048, need);
        } else {
            for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[0][i] = 0;
            __syncthreads();
            for (int64_t base = lo; base < hi; base += (int64_t)TK_T * TK_V) {
                uint32_t key[TK_V];
                int64_t pos[TK_V / 4];
                load_keys(sc, base, hi, vec, key, pos);
#pragma unroll
                for (int e = 0; e < TK_V; ++e) hist_add(sm.hist[0], key[e] >> 21, pos[e / 4] + (e & 3) < hi);
            }
            cluster_sync();
            find_bin(sm, HIST_CLUSTER, nullptr, 0, 2048, need);
        }
        const uint32_t b0 = sm.bin;
        need -= sm.above;
        // ---- 2. one scan of the slice: winners (digit > b0) and survivors (digit == b0)
        for (int64_t base = lo; base < hi; base += (int64_t)TK_T * TK_V) {
            uint32_t key[TK_V];
            int64_t pos[TK_V / 4];
            load_keys(sc, base, hi, vec, key, pos);
            uint32_t ns = 0, nc = 0;
#pragma unroll
            for (int e = 0; e < TK_V; ++e) {
                const bool in = pos[e / 4] + (e & 3) < hi;
                const uint32_t d = key[e] >> 21;
                ns += (in && d > b0) ? 1u : 0u;
                nc += (in && d == b0) ? 1u : 0u;
            }
            if (!__any_sync(0xffffffffu, (ns | nc) != 0)) continue;
            int bs, bc;
            warp_reserve(&sm.n_sel, &sm.n_cand, ns, nc, bs, bc);
#pragma unroll
            for (int e = 0; e < TK_V; ++e) {
                const int64_t i = pos[e / 4] + (e & 3);
                const bool in = i < hi;
                const uint32_t d = key[e] >> 21;
                if (in && d > b0) {
                    if (bs < TK_KMAX) { sm.skey[bs] = key[e]; sm.sidx[bs] = (int32_t)i; }
                    ++bs;
                } else if (in && d == b0) {
                    if (bc < TK_CAP) { sm.ckey[bc] = key[e]; sm.cidx[bc] = (int32_t)i; }
                    else sm.overflow = 1;
                    ++bc;
                }
            }
        }
        __syncthreads();
        // ---- 3. digits bits 20..10 and 9..0, refined across the cluster.  After the first of
        //      them the survivors normally fit CTA 0, which then finishes alone.
        uint32_t prefix = b0;
        int prev_shift = 21;
        const int shifts[2] = {10, 0};
        const int widths[2] = {11, 10};
        for (int p = 0; p < 2; ++p) {
            const int shift = shifts[p];
            const uint32_t mask = (1u << widths[p]) - 1u;
            const int nbins = 1 << widths[p];
            const int hb = (p + 1) & 1;
            for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[hb][i] = 0;
            __syncthreads();
            const bool list_mode = !sm.overflow;
            const int n_list = sm.n_cand;
            if (list_mode) {
                for (int i0 = 0; i0 < n_list; i0 += TK_T) {
                    const int i = i0 + tid;
                    const bool in = i < n_list;
                    const uint32_t key = in ? sm.ckey[i] : 0u;
                    hist_add(sm.hist[hb], (key >> shift) & mask, in);
                }
            } else {
                for (int64_t base = lo; base < hi; base += (int64_t)TK_T * TK_V) {
                    uint32_t key[TK_V];
                    int64_t pos[TK_V / 4];
                    load_keys(sc, base, hi, vec, key, pos);
#pragma unroll
                    for (int e = 0; e < TK_V; ++e) {
                        const bool in = pos[e / 4] + (e & 3) < hi && (key[e] >> prev_shift) == prefix;
                        hist_add(sm.hist[hb], (key[e] >> shift) & mask, in);
                    }
                }
            }
            cluster_sync();
            find_bin(sm, HIST_CLUSTER, nullptr, hb, nbins, need);
            const uint32_t bin = sm.bin;
            need -= sm.above;
            if (list_mode) {
                if (tid == 0) sm.n_new = 0;
                __syncthreads();
                for (int i0 = 0; i0 < n_list; i0 += TK_T) {
                    const int i = i0 + tid;
                    const bool in = i < n_list;
                    const uint32_t key = in ? sm.ckey[i] : 0u;
                    const int32_t idx = in ? sm.cidx[i] : 0;
                    __syncthreads();  // chunk read by everyone before it is overwritten
                    const uint32_t d = (key >> shift) & mask;
                    const int s = warp_alloc(&sm.n_sel, in && d > bin);
                    if (s >= 0 && s < TK_KMAX) { sm.skey[s] = key; sm.sidx[s] = idx; }
                    const int c = warp_alloc(&sm.n_new, in && d == bin);
                    if (c >= 0) { sm.ckey[c] = key; sm.cidx[c] = idx; }
                }
                __syncthreads();
                if (tid == 0) sm.n_cand = sm.n_new;
            } else {
                if (tid == 0) { sm.n_cand = 0; sm.overflow = 0; }
                __syncthreads();
                for (int64_t base = lo; base < hi; base += (int64_t)TK_T * TK_V) {
                    uint32_t key[TK_V];
                    int64_t pos[TK_V / 4];
                    load_keys(sc, base, hi, vec, key, pos);
#pragma unroll
                    for (int e = 0; e < TK_V; ++e) {
                        const int64_t i = pos[e / 4] + (e & 3);
                        const bool in = i < hi && (key[e] >> prev_shift) == prefix;
                        const uint32_t d = (key[e] >> shift) & mask;
                        const int s = warp_alloc(&sm.n_sel, in && d > bin);
                        if (s >= 0 && s < TK_KMAX) { sm.skey[s] = key[e]; sm.sidx[s] = (int32_t)i; }
                        const int c = warp_alloc(&sm.n_cand, in && d == bin);
                        if (c >= TK_CAP) sm.overflow = 1;
                        else if (c >= 0) { sm.ckey[c] = key[e]; sm.cidx[c] = (int32_t)i; }
                    }
                }
            }
            __syncthreads();
            prefix = (prefix << widths[p]) | bin;
            prev_shift = shift;
            if (p != 0) continue;
            // ---- exchange the counts; fast finish in CTA 0 when the survivors fit
            if (tid == 0) {
                sm.xchg[0] = (uint32_t)sm.n_sel;
                sm.xchg[1] = sm.overflow ? 0xFFFFFFFFu : (uint32_t)sm.n_cand;
            }
            cluster_sync();
            uint32_t off_sel = 0, tot_sel = 0, off_cand = 0, tot_cand = 0;
            bool any_over = false;
            for (uint32_t c = 0; c < TK_CL; ++c) {
                const uint32_t ns = ld_dsmem_u32(mapa(smem_u32(&sm.xchg[0]), c));
                const uint32_t nc = ld_dsmem_u32(mapa(smem_u32(&sm.xchg[1]), c));
                if (nc == 0xFFFFFFFFu) any_over = true;
                if (c < rank) { off_sel += ns; off_cand += nc; }
                tot_sel += ns;
                tot_cand += nc;
            }
            if (any_over || tot_cand > (uint32_t)TK_GCAP) continue;  // keep refining across the cluster
            for (int i = tid; i < sm.n_sel; i += TK_T) {
                st_dsmem_u32(mapa(smem_u32(&sm.okey[off_sel + i]), 0), sm.skey[i]);
                st_dsmem_u32(mapa(smem_u32(&sm.oidx[off_sel + i]), 0), (uint32_t)sm.sidx[i]);
            }
            for (int i = tid; i < sm.n_cand; i += TK_T) {
                st_dsmem_u32(mapa(smem_u32(&sm.gkey[off_cand + i]), 0), sm.ckey[i]);
                st_dsmem_u32(mapa(smem_u32(&sm.gidx[off_cand + i]), 0), (uint32_t)sm.cidx[i]);
            }
            cluster_sync();
            if (rank != 0) return;
            if (tid == 0) sm.n_out = (int)tot_sel;
            __syncthreads();
            int n_list2 = (int)tot_cand;
            if (n_list2 > TK_T && (uint32_t)n_list2 != need) {
                // last digit (bits 9..0) locally, then the ties
                for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[0][i] = 0;
                __syncthreads();
                for (int i0 = 0; i0 < n_list2; i0 += TK_T) {
                    const int i = i0 + tid;
                    const bool in = i < n_list2;
                    hist_add(sm.hist[0], in ? (sm.gkey[i] & 1023u) : 0u, in);
                }
                __syncthreads();
                find_bin(sm, HIST_LOCAL, nullptr, 0, 1024, need);
                const uint32_t lbin = sm.bin;
                need -= sm.above;
                if (tid == 0) sm.n_new = 0;
                __syncthreads();
                for (int i0 = 0; i0 < n_list2; i0 += TK_T) {
                    const int i = i0 + tid;
                    const bool in = i < n_list2;
                    const uint32_t key = in ? sm.gkey[i] : 0u;
                    const int32_t idx = in ? sm.gidx[i] : 0;
                    __syncthreads();
                    const uint32_t d = key & 1023u;
                    const int so = warp_alloc(&sm.n_out, in && d > lbin);
                    if (so >= 0 && so < TK_KMAX) { sm.okey[so] = key; sm.oidx[so] = idx; }
                    const int c = warp_alloc(&sm.n_new, in && d == lbin);
                    if (c >= 0) { sm.gkey[c] = key; sm.gidx[c] = idx; }
                }
                __syncthreads();
                n_list2 = sm.n_new;
            }
            // the `need` best survivors by (key desc, index asc): rank each against all
            for (int i = tid; i < n_list2; i += TK_T) {
                const uint32_t myk = sm.gkey[i];
                const int32_t myi = sm.gidx[i];
                uint32_t rnk = 0;
                for (int j = 0; j < n_list2; ++j) rnk += kv_greater(sm.gkey[j], sm.gidx[j], myk, myi) ? 1u : 0u;
                if (rnk < need) {
                    const int so = atomicAdd(&sm.n_out, 1);
                    if (so < TK_KMAX) { sm.okey[so] = myk; sm.oidx[so] = myi; }
                }
            }
            __syncthreads();
            sort_and_write(sm, (uint32_t)min(sm.n_out, k), k, out, kout);
            return;
        }
        // prefix == tau (full key); `need` ties at tau remain to be taken, lowest index first.
        const uint32_t tau = prefix;
        const bool list_mode = !sm.overflow;
        if (!list_mode) {
            if (tid == 0) sm.cnt = 0;
            __syncthreads();
            for (int64_t i0 = lo; i0 < hi; i0 += TK_T) {
                const int64_t i = i0 + tid;
                const bool f = i < hi && score_key(__ldg(sc + i)) == tau;
                warp_alloc(reinterpret_cast<int*>(&sm.cnt), f);
            }
            __syncthreads();
        } else if (tid == 0) {
            sm.cnt = (uint32_t)sm.n_cand;
        }
        __syncthreads();
        const uint32_t c_r = sm.cnt;
        if (tid == 0) sm.xchg[2] = c_r;
        cluster_sync();
        uint32_t before = 0;
        for (uint32_t c = 0; c < rank; ++c) before += ld_dsmem_u32(mapa(smem_u32(&sm.xchg[2]), c));
        const uint32_t take = need > before ? min(need - before, c_r) : 0u;
        if (take > 0) {
            if (take == c_r && list_mode) {
                for (int i = tid; i < (int)c_r; i += TK_T) {
                    const int s = atomicAdd(&sm.n_sel, 1);
                    if (s < TK_KMAX) { sm.skey[s] = tau; sm.sidx[s] = sm.cidx[i]; }
                }
            } else if (list_mode && c_r <= (uint32_t)TK_T) {
                if (tid < (int)c_r) {
                    const int32_t my = sm.cidx[tid];
                    uint32_t rnk = 0;
                    for (uint32_t j = 0; j < c_r; ++j) rnk += sm.cidx[j] < my ? 1u : 0u;
                    if (rnk < take) {
                        const int s = atomicAdd(&sm.n_sel, 1);
                        if (s < TK_KMAX) { sm.skey[s] = tau; sm.sidx[s] = my; }
                    }
                }
            } else {
                // ordered scan of the slice: the first `take` ties in index order
                if (tid == 0) sm.taken = 0;
                __syncthreads();
                for (int64_t i0 = lo; i0 < hi; i0 += TK_T) {
                    const int64_t i = i0 + tid;
                    const bool f = i < hi && score_key(__ldg(sc + i)) == tau;
                    uint32_t tot;
                    const uint32_t ex = block_scan(sm, f ? 1u : 0u, &tot);
                    const uint32_t base = sm.taken;
                    if (f && base + ex < take) {
                        const int s = atomicAdd(&sm.n_sel, 1);
                        if (s < TK_KMAX) { sm.skey[s] = tau; sm.sidx[s] = (int32_t)i; }
                    }
                    __syncthreads();
                    if (tid == 0) sm.taken = base + tot;
                    __syncthreads();
                    if (sm.taken >= take) break;
                }
            }
        }
        __syncthreads();
    } else {
        // every candidate is selected
        for (int64_t i0 = lo; i0 < hi; i0 += TK_T) {
            const int64_t i = i0 + tid;
            const bool in = i < hi;
            const uint32_t key = in ? score_key(__ldg(sc + i)) : 0u;
            const int s = warp_alloc(&sm.n_sel, in);
            if (s >= 0 && s < TK_KMAX) { sm.skey[s] = key; sm.sidx[s] = (int32_t)i; }
        }
        __syncthreads();
    }

    // ---- gather the cluster's winners into CTA 0 (cluster-wide path)
    const uint32_t n_mine = (uint32_t)min(sm.n_sel, TK_KMAX);
    if (tid == 0) {
        sm.xchg[3] = n_mine;
        if (sm.n_sel > TK_KMAX) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    }
    cluster_sync();
    uint32_t off = 0, total = 0;
    for (uint32_t c = 0; c < TK_CL; ++c) {
        const uint32_t v = ld_dsmem_u32(mapa(smem_u32(&sm.xchg[3]), c));
        if (c < rank) off += v;
        total += v;
    }
    for (uint32_t i = tid; i < n_mine; i += TK_T) {
        if (off + i < (uint32_t)TK_KMAX) {
            st_dsmem_u32(mapa(smem_u32(&sm.okey[off + i]), 0), sm.skey[i]);
            st_dsmem_u32(mapa(smem_u32(&sm.oidx[off + i]), 0), (uint32_t)sm.sidx[i]);
        }
    }
    cluster_sync();
    if (rank != 0) return;
    sort_and_write(sm, total, k, out, kout);
}

cudaError_t launch_topk(const TopkLaunch& h, cudaStream_t s, bool pdl) {
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
    a.status = h.status;
    const size_t smem = sizeof(TkSmem);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = TK_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    cfg.gridDim = dim3((unsigned)(TK_CL * h.B), 1, 1);
    cfg.blockDim = dim3(TK_T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, topk_kernel, a);
}

}  // namespace csa
