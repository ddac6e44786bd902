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
// [r*S, r*S+S).  Digits of the key: bits 31..21, 20..10, 9..0.  For each digit
// every CTA builds a local histogram of the candidates that still match the
// prefix, the 8 histograms are summed through distributed shared memory, and
// every CTA finds the same bin that contains the k-th key.  Entries in higher
// bins are selected; the matching bin's entries survive (kept in shared memory,
// or re-read from L2 when more than CAP survive).  In the fused decode step the
// first digit's histogram comes ready from the score kernel, so the first pass
// is a single filtered scan.  After the last digit tau is exact; ties at tau are
// taken lowest index first (slices are in index order across the cluster).  CTA
// 0 gathers the k winners through DSMEM and sorts them (bitonic, shared memory).
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int TK_CL = 8;
constexpr int TK_T = 1024;
constexpr int TK_BINS = kHistBins;   // 2048: widest digit
constexpr int TK_CAP = 12288;
constexpr int TK_KMAX = 2048;
constexpr int TK_U = 4;              // independent loads in flight per thread in the scans

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
    uint32_t ckey[TK_CAP];
    int32_t cidx[TK_CAP];
    uint32_t skey[TK_KMAX];
    int32_t sidx[TK_KMAX];
    uint32_t okey[TK_KMAX];
    int32_t oidx[TK_KMAX];
    uint32_t xchg[4];
    uint32_t wsum[32];
    int n_cand, n_sel, n_new, overflow;
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

// Total histogram (the global one from the score kernel, or the sum of the 8
// CTAs' through DSMEM), then the bin holding the need-th largest key counted from
// the top bin.  Writes sm.bin and sm.above (count in higher bins).
__device__ __forceinline__ void reduce_and_find(TkSmem& sm, const uint32_t* ghist, int hb, int nbins,
                                                uint32_t need) {
    const int t = threadIdx.x;
    const int bh = nbins - 1 - 2 * t, bl = nbins - 2 - 2 * t;  // this thread's two bins, high first
    uint32_t th = 0, tl = 0;
    if (bl >= 0) {
        if (ghist) {
            th = __ldg(ghist + bh);
            tl = __ldg(ghist + bl);
        } else {
            const uint32_t ah = smem_u32(&sm.hist[hb][bh]), al = smem_u32(&sm.hist[hb][bl]);
#pragma unroll
            for (int c = 0; c < TK_CL; ++c) {
                th += ld_dsmem_u32(mapa(ah, c));
                tl += ld_dsmem_u32(mapa(al, c));
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

__device__ __forceinline__ bool kv_greater(uint32_t ka, int32_t ia, uint32_t kb, int32_t ib) {
    return ka > kb || (ka == kb && ia < ib);
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
    const int64_t slice = (G + TK_CL - 1) / TK_CL;
    const int64_t lo = min((int64_t)rank * slice, G), hi = min(lo + slice, G);
    const uint32_t need_total = (uint32_t)min((int64_t)k, G);

    if (tid == 0) {
        sm.n_cand = 0;
        sm.n_sel = 0;
        sm.overflow = 0;
    }
    __syncthreads();

    if (G > k) {
        const int shifts[3] = {21, 10, 0};
        const int widths[3] = {11, 11, 10};
        uint32_t need = need_total;
        uint32_t prefix = 0;
        int prev_shift = 32;
        for (int p = 0; p < 3; ++p) {
            const int shift = shifts[p];
            const uint32_t mask = (1u << widths[p]) - 1u;
            const int nbins = 1 << widths[p];
            const int hb = p & 1;
            const bool fused = p == 0 && a.hist != nullptr;
            const uint32_t* gh = fused ? a.hist + (int64_t)b * kHistBins : nullptr;
            if (!fused)
                for (int i = tid; i < TK_BINS; i += TK_T) sm.hist[hb][i] = 0;
            __syncthreads();
            const bool list_mode = p > 0 && !sm.overflow;
            const int n_list = sm.n_cand;
            // ---- histogram of the surviving candidates
            if (!fused) {
                if (list_mode) {
                    for (int i0 = 0; i0 < n_list; i0 += TK_T) {
                        const int i = i0 + tid;
                        const bool in = i < n_list;
                        const uint32_t key = in ? sm.ckey[i] : 0u;
                        hist_add(sm.hist[hb], (key >> shift) & mask, in);
                    }
                } else {
                    for (int64_t i0 = lo; i0 < hi; i0 += TK_U * TK_T) {
                        uint32_t key[TK_U];
                        bool in[TK_U];
#pragma unroll
                        for (int u = 0; u < TK_U; ++u) {
                            const int64_t i = i0 + u * TK_T + tid;
                            in[u] = i < hi;
                            key[u] = in[u] ? score_key(__ldg(sc + i)) : 0u;
                            if (prev_shift < 32) in[u] = in[u] && (key[u] >> prev_shift) == prefix;
                        }
#pragma unroll
                        for (int u = 0; u < TK_U; ++u) hist_add(sm.hist[hb], (key[u] >> shift) & mask, in[u]);
                    }
                }
                cluster_sync();
            }
            reduce_and_find(sm, gh, hb, nbins, need);
            const uint32_t bin = sm.bin;
            need -= sm.above;
            // ---- select the higher bins, keep the matching bin
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
                for (int64_t i0 = lo; i0 < hi; i0 += TK_U * TK_T) {
                    uint32_t key[TK_U], d[TK_U];
                    bool in[TK_U];
                    bool mine = false;
#pragma unroll
                    for (int u = 0; u < TK_U; ++u) {
                        const int64_t i = i0 + u * TK_T + tid;
                        in[u] = i < hi;
                        key[u] = in[u] ? score_key(__ldg(sc + i)) : 0u;
                        if (prev_shift < 32) in[u] = in[u] && (key[u] >> prev_shift) == prefix;
                        d[u] = (key[u] >> shift) & mask;
                        mine = mine || (in[u] && d[u] >= bin);
                    }
                    if (!__any_sync(0xffffffffu, mine)) continue;  // nothing at or above the bin here
#pragma unroll
                    for (int u = 0; u < TK_U; ++u) {
                        const int32_t idx = (int32_t)(i0 + u * TK_T + tid);
                        const int s = warp_alloc(&sm.n_sel, in[u] && d[u] > bin);
                        if (s >= 0 && s < TK_KMAX) { sm.skey[s] = key[u]; sm.sidx[s] = idx; }
                        const int c = warp_alloc(&sm.n_cand, in[u] && d[u] == bin);
                        if (c >= TK_CAP) sm.overflow = 1;
                        else if (c >= 0) { sm.ckey[c] = key[u]; sm.cidx[c] = idx; }
                    }
                }
            }
            __syncthreads();
            prefix = (prev_shift < 32 ? (prefix << widths[p]) : 0u) | bin;
            prev_shift = shift;
        }
        // prefix == tau (full key); `need` ties at tau remain to be taken.
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
        if (tid == 0) sm.xchg[0] = c_r;
        cluster_sync();
        uint32_t before = 0;
        for (uint32_t c = 0; c < rank; ++c) before += ld_dsmem_u32(mapa(smem_u32(&sm.xchg[0]), c));
        const uint32_t take = need > before ? min(need - before, c_r) : 0u;
        if (take > 0) {
            if (take == c_r && list_mode) {
                for (int i = tid; i < (int)c_r; i += TK_T) {
                    const int s = atomicAdd(&sm.n_sel, 1);
                    if (s < TK_KMAX) { sm.skey[s] = tau; sm.sidx[s] = sm.cidx[i]; }
                }
            } else if (list_mode && c_r <= (uint32_t)TK_T) {
                // rank of each tie among this CTA's ties by index; keep the `take` lowest
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

    // ---- gather the cluster's selections into CTA 0
    const uint32_t n_mine = (uint32_t)min(sm.n_sel, TK_KMAX);
    if (tid == 0) {
        sm.xchg[1] = n_mine;
        if (sm.n_sel > TK_KMAX) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    }
    cluster_sync();
    uint32_t off = 0, total = 0;
    for (uint32_t c = 0; c < TK_CL; ++c) {
        const uint32_t v = ld_dsmem_u32(mapa(smem_u32(&sm.xchg[1]), c));
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

    // ---- CTA 0: bitonic sort of the winners by (key desc, index asc)
    if (total > (uint32_t)TK_KMAX) total = TK_KMAX;
    int n2 = 1;
    while (n2 < (int)total) n2 <<= 1;
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
                    const bool first_half = (i & size) == 0;  // this block is sorted "greater first"
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
    int32_t* out = a.idx_out + (int64_t)b * k;
    uint32_t* kout = a.keys_out ? a.keys_out + (int64_t)b * k : nullptr;
    for (int i = tid; i < k; i += TK_T) {
        const bool v = i < (int)total;
        out[i] = v ? sm.oidx[i] : -1;
        if (kout) kout[i] = v ? sm.okey[i] : 0u;
    }
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
