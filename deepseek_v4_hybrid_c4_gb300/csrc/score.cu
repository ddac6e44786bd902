// Stage 2: indexer score of every compressed candidate ("DeepSeek-V4 本地部署，SGLang
// 把活做絕了", sec. "Kernel 層一堆狠活": 256K candidates at 1M context feed the top-512).
//
//   score[g] = sum_h w_h * ReLU(q_idx[h] . k_idx[g])     fp32, bit-exact fixed order:
//   P[t]  = q[8t]*k[8t], then fma over dims 8t+1..8t+7   (chunk t = 0..15, one lane each)
//   S1[t] = P[t] + P[t+8]; S2 = S1[t] + S1[t+4]; S3 = S2[t] + S2[t+2]; dot = S3[0] + S3[1]
//   acc = fma(w_h, ReLU(dot_h), acc) for h = 0..Hi-1, from acc = 0
//
// Layout: a candidate row (128 dims: 256 B bf16 / 128 B fp8) is owned by a
// half-warp; lane t holds chunk t (one 16-byte / 8-byte shared load) and the
// index query q_idx[.][8t..8t+7] stays in registers, packed as head pairs so each
// packed fma.rn.f32x2 advances two heads' chains (two IEEE fmas: exactness holds).
// The butterfly runs as a reduce-scatter over the heads with shuffle masks 8, 4,
// 2, 1 (Hi/2 + Hi/4 + ... shuffles per two rows).  Each consumer warp works on
// two row pairs at once so the shuffle latency of one hides behind the other.
//
// Memory path: a producer lane streams 16-row units (one unit never crosses a
// page) with cp.async.bulk into a ring of shared-memory stages tracked by
// mbarriers; 4 consumer warps drain it.  Persistent grid, 3 CTAs per SM: one
// long stream of 4 KiB (bf16) / 2 KiB (fp8) pieces through HBM.
//
// Optional fused epilogue: a histogram of the top 11 bits of each score's
// order-preserving key (the first digit of the top-k radix select), per request,
// accumulated in shared memory and added to a global [B][2048] histogram.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int SC_CONSUMERS = 4;              // consumer warps, 4 rows each per 16-row unit
constexpr int SC_THREADS = (SC_CONSUMERS + 1) * 32;
constexpr int SC_UNIT = 16;                  // rows per unit
constexpr int SC_STAGES = 8;

struct ScoreArgs {
    const uint16_t* q_idx;
    const float* w_h;
    int Hi;
    DPaged kidx;
    float* scores;
    int64_t score_stride;
    int B;
    const int64_t* n_tokens;
    int ratio;
    int64_t G;
    uint32_t* hist;          // [B][kHistBins] or nullptr
    int32_t* status;
};

// Walks the concatenated unit space of the batch: after seek(w), unit w belongs
// to request b, whose candidates number G.  Returns false past the end.
struct UnitCursor {
    int b = -1;
    int64_t base = 0, units = 0, G = 0;
    __device__ void load(const ScoreArgs& a) {
        G = a.n_tokens ? __ldg(a.n_tokens + b) / a.ratio : a.G;
        units = (G + SC_UNIT - 1) / SC_UNIT;
    }
    __device__ bool seek(const ScoreArgs& a, int64_t w) {
        if (b < 0) {
            if (a.B <= 0) return false;
            b = 0;
            load(a);
        }
        while (w >= base + units) {
            base += units;
            if (++b >= a.B) return false;
            load(a);
        }
        return true;
    }
};

__device__ __forceinline__ void fp8x8_to_f32(uint2 raw, float (&k)[8]) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h01, h23;
        const uint16_t lo = (uint16_t)(w[i] & 0xFFFFu), hi = (uint16_t)(w[i] >> 16);
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"(lo));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"(hi));
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 fc = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        k[4 * i + 0] = fa.x;
        k[4 * i + 1] = fa.y;
        k[4 * i + 2] = fc.x;
        k[4 * i + 3] = fc.y;
    }
}

__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// One reduce-scatter stage over C head values with shuffle mask MASK.
template <int C, int MASK>
__device__ __forceinline__ void rs_stage(float (&v)[16], int lane, int& head_base) {
    if constexpr (C >= 2) {
        const bool upper = (lane & MASK) != 0;
#pragma unroll
        for (int h = 0; h < C / 2; ++h) {
            const float send = upper ? v[h] : v[h + C / 2];
            const float keep = upper ? v[h + C / 2] : v[h];
            v[h] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
        }
        if (upper) head_base += C / 2;
    } else {
        v[0] = v[0] + __shfl_xor_sync(0xffffffffu, v[0], MASK);
    }
}

template <int HI>
__device__ __forceinline__ int head_dots(const uint64_t (&qp)[HI / 2][8], const float (&k)[8], float (&v)[16],
                                         int lane) {
    uint64_t acc[HI / 2];
#pragma unroll
    for (int hp = 0; hp < HI / 2; ++hp) acc[hp] = mul2(qp[hp][0], pk2(k[0], k[0]));
#pragma unroll
    for (int e = 1; e < 8; ++e) {
        const uint64_t kk = pk2(k[e], k[e]);
#pragma unroll
        for (int hp = 0; hp < HI / 2; ++hp) acc[hp] = fma2(qp[hp][e], kk, acc[hp]);
    }
#pragma unroll
    for (int hp = 0; hp < HI / 2; ++hp) {
        v[2 * hp] = __uint_as_float((uint32_t)acc[hp]);
        v[2 * hp + 1] = __uint_as_float((uint32_t)(acc[hp] >> 32));
    }
    int hb = 0;
    rs_stage<HI, 8>(v, lane, hb);
    rs_stage<(HI >= 2 ? HI / 2 : 1), 4>(v, lane, hb);
    rs_stage<(HI >= 4 ? HI / 4 : 1), 2>(v, lane, hb);
    rs_stage<(HI >= 8 ? HI / 8 : 1), 1>(v, lane, hb);
    return hb;
}

template <bool FP8>
__device__ __forceinline__ void load_row_chunk(const uint8_t* stage, int row, int t, bool valid, float (&k)[8]) {
    constexpr int RB = FP8 ? 128 : 256;
    if (valid) {
        const uint32_t addr = smem_u32(stage + row * RB + t * (FP8 ? 8 : 16));
        if constexpr (FP8) {
            fp8x8_to_f32(ld_shared_v2(addr), k);
        } else {
            const uint4 r = ld_shared_v4(addr);
            k[0] = bf16lo(r.x); k[1] = bf16hi(r.x); k[2] = bf16lo(r.y); k[3] = bf16hi(r.y);
            k[4] = bf16lo(r.z); k[5] = bf16hi(r.z); k[6] = bf16lo(r.w); k[7] = bf16hi(r.w);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) k[e] = 0.f;
    }
}

__device__ __forceinline__ void consumer_bar() { asm volatile("bar.sync 1, %0;" ::"n"(SC_CONSUMERS * 32) : "memory"); }

template <int HI, bool FP8>
__global__ void __launch_bounds__(SC_THREADS, HI <= 8 ? 3 : 1) score_kernel(ScoreArgs a) {
    constexpr int RB = FP8 ? 128 : 256;          // bytes per candidate row
    constexpr int STAGE_BYTES = SC_UNIT * RB;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SC_STAGES * STAGE_BYTES);
    uint64_t* empty = full + SC_STAGES;
    int* meta = reinterpret_cast<int*>(empty + SC_STAGES);          // page valid flag per stage
    float* red = reinterpret_cast<float*>(meta + SC_STAGES);        // [warp][pair][half][HI]
    uint32_t* hist = reinterpret_cast<uint32_t*>(red + SC_CONSUMERS * 4 * HI);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (a.hist)
        for (int i = threadIdx.x; i < kHistBins; i += SC_THREADS) hist[i] = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), SC_CONSUMERS);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == SC_CONSUMERS) {
        // ---------------- producer: one lane issues the bulk copies
        if (lane == 0) {
            UnitCursor cur;
            for (int64_t i = 0;; ++i) {
                const int64_t w = blockIdx.x + i * gridDim.x;
                if (!cur.seek(a, w)) break;
                const int s = (int)(i % SC_STAGES);
                if (i >= SC_STAGES && !mbar_wait(smem_u32(&empty[s]), (uint32_t)(((i / SC_STAGES) - 1) & 1))) {
                    raise_status(a.status, CSA_ERR_TIMEOUT);
                    break;
                }
                const int64_t g0 = (w - cur.base) * SC_UNIT;
                const int nrows = (int)(cur.G - g0 < SC_UNIT ? cur.G - g0 : SC_UNIT);
                const uint8_t* src = row_addr(a.kidx, cur.b, g0, RB, a.status);
                meta[s] = src ? 1 : 0;
                const uint32_t fb = smem_u32(&full[s]);
                if (src) {
                    mbar_arrive_expect_tx(fb, (uint32_t)(nrows * RB));
                    bulk_g2s(smem_u32(stages + s * STAGE_BYTES), src, (uint32_t)(nrows * RB), fb);
                } else {
                    mbar_arrive(fb);
                }
            }
        }
        return;
    }

    // ---------------- consumers
    const int t = lane & 15;            // chunk: dims 8t .. 8t+7
    const int half = lane >> 4;         // row within a pair
    uint64_t qp[HI / 2][8];
    float wv[HI];
    int qb = -1;
    float* my_red = red + warp * 4 * HI;
    UnitCursor cur;
    for (int64_t i = 0;; ++i) {
        const int64_t w = blockIdx.x + i * gridDim.x;
        if (!cur.seek(a, w)) break;
        const int s = (int)(i % SC_STAGES);
        if (cur.b != qb) {
            if (a.hist && qb >= 0) {  // flush the finished request's histogram
                consumer_bar();
                for (int bin = threadIdx.x; bin < kHistBins; bin += SC_CONSUMERS * 32) {
                    const uint32_t c = hist[bin];
                    if (c) {
                        atomicAdd(a.hist + (int64_t)qb * kHistBins + bin, c);
                        hist[bin] = 0;
                    }
                }
                consumer_bar();
            }
            qb = cur.b;
            const uint16_t* qptr = a.q_idx + (int64_t)qb * a.Hi * DI;
#pragma unroll
            for (int hp = 0; hp < HI / 2; ++hp) {
                float q0[8], q1[8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int h = 2 * hp + u;
                    float* qq = u ? q1 : q0;
                    if (h < a.Hi) {
                        const uint4 r = __ldg(reinterpret_cast<const uint4*>(qptr + h * DI + 8 * t));
                        qq[0] = bf16lo(r.x); qq[1] = bf16hi(r.x); qq[2] = bf16lo(r.y); qq[3] = bf16hi(r.y);
                        qq[4] = bf16lo(r.z); qq[5] = bf16hi(r.z); qq[6] = bf16lo(r.w); qq[7] = bf16hi(r.w);
                        wv[h] = __ldg(a.w_h + (int64_t)qb * a.Hi + h);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) qq[e] = 0.f;
                        wv[h] = 0.f;
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) qp[hp][e] = pk2(q0[e], q1[e]);
            }
        }
        if (!mbar_wait(smem_u32(&full[s]), (uint32_t)((i / SC_STAGES) & 1))) {
            raise_status(a.status, CSA_ERR_TIMEOUT);
            break;
        }
        const int64_t g0 = (w - cur.base) * SC_UNIT;
        const int nrows = (int)(cur.G - g0 < SC_UNIT ? cur.G - g0 : SC_UNIT);
        const int page_ok = meta[s];
        const int rowA = 4 * warp + half, rowB = 4 * warp + 2 + half;
        float kA[8], kB[8];
        const uint8_t* st = stages + s * STAGE_BYTES;
        load_row_chunk<FP8>(st, rowA, t, page_ok && rowA < nrows, kA);
        load_row_chunk<FP8>(st, rowB, t, page_ok && rowB < nrows, kB);
        // the stage's bytes are in registers: release it to the producer
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        float vA[16], vB[16];
        const int hA = head_dots<HI>(qp, kA, vA, lane);
        const int hB = head_dots<HI>(qp, kB, vB, lane);
        // lane holds the dot of head hA (row A) / hB (row B); ReLU, then the head chain in order
        my_red[(0 * 2 + half) * HI + hA] = vA[0] > 0.f ? vA[0] : 0.f;
        my_red[(1 * 2 + half) * HI + hB] = vB[0] > 0.f ? vB[0] : 0.f;
        __syncwarp();
        if (t < 2) {  // lane t = 0 finishes row A, lane t = 1 row B
            const int pr = t;
            const int row = 4 * warp + 2 * pr + half;
            float acc = 0.f;
#pragma unroll
            for (int h = 0; h < HI; ++h) acc = __fmaf_rn(wv[h], my_red[(pr * 2 + half) * HI + h], acc);
            if (row < nrows) {
                const float sc = page_ok ? acc : 0.f;
                a.scores[(int64_t)cur.b * a.score_stride + g0 + row] = sc;
                if (a.hist) atomicAdd(&hist[score_key(sc) >> 21], 1u);
            }
        }
        __syncwarp();
    }
    if (a.hist && qb >= 0) {
        consumer_bar();
        for (int bin = threadIdx.x; bin < kHistBins; bin += SC_CONSUMERS * 32) {
            const uint32_t c = hist[bin];
            if (c) atomicAdd(a.hist + (int64_t)qb * kHistBins + bin, c);
        }
    }
}

template <int HI, bool FP8>
static cudaError_t launch_score_t(const ScoreArgs& a, int64_t total_units_bound, cudaStream_t s, bool pdl) {
    constexpr int RB = FP8 ? 128 : 256;
    constexpr size_t base = (size_t)SC_STAGES * SC_UNIT * RB + 2 * SC_STAGES * sizeof(uint64_t) +
                            SC_STAGES * sizeof(int) + SC_CONSUMERS * 4 * HI * sizeof(float);
    const size_t smem = base + (a.hist ? kHistBins * sizeof(uint32_t) : 0);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(score_kernel<HI, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(base + kHistBins * sizeof(uint32_t)));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    int64_t grid = (HI <= 8 ? 3LL : 1LL) * sms;
    if (total_units_bound < grid) grid = total_units_bound < 1 ? 1 : total_units_bound;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(SC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, score_kernel<HI, FP8>, a);
}

cudaError_t launch_score(const ScoreLaunch& h, cudaStream_t s, bool pdl) {
    ScoreArgs a;
    a.q_idx = static_cast<const uint16_t*>(h.q_idx);
    a.w_h = h.w_h;
    a.Hi = h.Hi;
    a.kidx.base = static_cast<const uint8_t*>(h.kidx.base);
    a.kidx.pt = h.kidx.pt;
    a.kidx.pt_stride = h.kidx.pt_stride;
    a.kidx.page_stride = h.kidx.page_stride;
    a.kidx.n_pages = h.kidx.n_pages;
    a.kidx.rpp = h.kidx.rpp;
    a.scores = h.scores;
    a.score_stride = h.score_stride;
    a.B = h.B;
    a.n_tokens = h.n_tokens;
    a.ratio = h.ratio;
    a.G = h.G;
    a.hist = h.hist;
    a.status = h.status;
    const int64_t units = (int64_t)h.B * ((h.max_G + SC_UNIT - 1) / SC_UNIT);
    const int hi = h.Hi <= 4 ? 4 : (h.Hi <= 8 ? 8 : 16);
    if (h.fp8) {
        if (hi == 4) return launch_score_t<4, true>(a, units, s, pdl);
        if (hi == 8) return launch_score_t<8, true>(a, units, s, pdl);
        return launch_score_t<16, true>(a, units, s, pdl);
    }
    if (hi == 4) return launch_score_t<4, false>(a, units, s, pdl);
    if (hi == 8) return launch_score_t<8, false>(a, units, s, pdl);
    return launch_score_t<16, false>(a, units, s, pdl);
}

}  // namespace csa
