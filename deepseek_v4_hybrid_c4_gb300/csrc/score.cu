// Stage 2: indexer score of every compressed candidate ("DeepSeek-V4 本地部署，SGLang
// 把活做絕了", sec. "Kernel 層一堆狠活": 256K candidates at 1M context feed the top-512).
//
//   score[g] = sum_h w_h * ReLU(q_idx[h] . k_idx[g])     fp32, bit-exact fixed order:
//   P[t]  = q[8t]*k[8t], then fma over dims 8t+1..8t+7   (chunk t = 0..15)
//   S1[t] = P[t] + P[t+8]; S2 = S1[t] + S1[t+4]; S3 = S2[t] + S2[t+2]; dot = S3[0] + S3[1]
//   acc = fma(w_h, ReLU(dot_h), acc) for h = 0..Hi-1, from acc = 0
//
// Layout: one candidate row per lane, so the whole fixed-order tree runs inside a
// lane with no shuffles.  A lane walks the chunk pairs (a, a+8) in bit-reversed
// order 0,4,2,6,1,5,3,7: each pair yields S1[a] with packed fma.rn.f32x2 (the two
// halves are the P[a] and P[a+8] chains -- two IEEE fmas per instruction), and the
// order makes every S2/S3 operand ready exactly when the tree needs it.  The
// index query is staged per warp in shared memory as {q[8a+i], q[8a+64+i]} pairs
// and read as broadcasts.
//
// Memory path: a producer lane streams 16-row units with TMA tensor copies
// (cp.async.bulk.tensor, 128-byte swizzle) into a ring of shared-memory stages
// tracked by mbarriers.  The swizzle puts 16-byte chunk c of row r at position
// c ^ (r & 7), so 32 lanes reading the same logical chunk of 32 different rows hit
// distinct banks.  A consumer warp takes two units (32 rows) at a time.
// Persistent grid, two CTAs per SM.
//
// Optional fused epilogue: a per-warp (16-bit) histogram of the top 11 bits of each score's
// order-preserving key (the first digit of the top-k radix select), flushed per
// request into a global [B][2048] histogram.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int SC_CONSUMERS = 4;              // consumer warps; each takes 32 rows (2 units) per step
constexpr int SC_THREADS = (SC_CONSUMERS + 1) * 32;
constexpr int SC_UNIT = 16;                  // rows per unit (one TMA box height)
constexpr int SC_SUPER = 32;                 // rows per consumer-warp step
constexpr int SC_STAGES = 18;                // units in flight per CTA
constexpr int SC_STAGE_BYTES = SC_UNIT * 256;  // bf16 unit (fp8 uses half)

struct ScoreArgs {
    const uint16_t* q_idx;
    const float* w_h;
    int Hi;
    const int32_t* pt;       // page table of the index-key pool (nullptr: contiguous rows)
    int64_t pt_stride;
    int64_t n_pages;
    int32_t rpp;             // rows per page (multiple of 16); contiguous: >= G
    float* scores;
    int64_t score_stride;
    int B;
    const int64_t* n_tokens;
    int ratio;
    int64_t G;
    uint32_t* hist;          // [B][kHistBins] or nullptr
    int32_t* status;
};

// Walks the concatenated space of 32-row steps of the batch (no step straddles two
// requests): after seek(w), step w belongs to request b, with G candidates.
struct StepCursor {
    int b = -1;
    int64_t base = 0, steps = 0, G = 0;
    __device__ void load(const ScoreArgs& a) {
        G = a.n_tokens ? __ldg(a.n_tokens + b) / a.ratio : a.G;
        steps = (G + SC_SUPER - 1) / SC_SUPER;
    }
    __device__ bool seek(const ScoreArgs& a, int64_t w) {
        if (b < 0) {
            if (a.B <= 0) return false;
            b = 0;
            load(a);
        }
        while (w >= base + steps) {
            base += steps;
            if (++b >= a.B) return false;
            load(a);
        }
        return true;
    }
};

__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
// Two {q_h[8a+i], q_h[8a+64+i]} pairs (heads h, h+1) straight into 64-bit registers.
__device__ __forceinline__ void ld_qpairs(uint32_t addr, uint64_t& p0, uint64_t& p1) {
    asm volatile("ld.shared.v2.u64 {%0, %1}, [%2];" : "=l"(p0), "=l"(p1) : "r"(addr));
}
__device__ __forceinline__ float lo2(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi2(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
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

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fp8x8(uint2 raw, float (&k)[8]) {
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h01, h23;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w[i] & 0xFFFFu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w[i] >> 16)));
        const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 fc = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        k[4 * i + 0] = fa.x;
        k[4 * i + 1] = fa.y;
        k[4 * i + 2] = fc.x;
        k[4 * i + 3] = fc.y;
    }
}

// The 16 key values of chunk pair (a, a+8) of the lane's row, from a swizzled stage.
template <bool FP8>
__device__ __forceinline__ void load_pair(const uint8_t* stage, int r, int a, float (&kl)[8], float (&kh)[8]) {
    const uint32_t base = smem_u32(stage) + (uint32_t)r * 128u;
    const uint32_t sw = (uint32_t)(r & 7);
    if constexpr (FP8) {
        // row = 128 fp8 = 8 chunks of 16 dims: dims 8a.. in chunk a/2, dims 64+8a.. in chunk 4+a/2
        const uint32_t off = (uint32_t)(a & 1) * 8u;
        fp8x8(ld_shared_v2(base + ((((uint32_t)a >> 1) ^ sw) << 4) + off), kl);
        fp8x8(ld_shared_v2(base + (((4u + ((uint32_t)a >> 1)) ^ sw) << 4) + off), kh);
    } else {
        // two 16-row boxes: dims 0..63 at +0, dims 64..127 at +2048; chunk a holds dims 8a..8a+7 of its half
        const uint4 x = ld_shared_v4(base + (((uint32_t)a ^ sw) << 4));
        const uint4 y = ld_shared_v4(base + 2048u + (((uint32_t)a ^ sw) << 4));
        kl[0] = bf16lo(x.x); kl[1] = bf16hi(x.x); kl[2] = bf16lo(x.y); kl[3] = bf16hi(x.y);
        kl[4] = bf16lo(x.z); kl[5] = bf16hi(x.z); kl[6] = bf16lo(x.w); kl[7] = bf16hi(x.w);
        kh[0] = bf16lo(y.x); kh[1] = bf16hi(y.x); kh[2] = bf16lo(y.y); kh[3] = bf16hi(y.y);
        kh[4] = bf16lo(y.z); kh[5] = bf16hi(y.z); kh[6] = bf16lo(y.w); kh[7] = bf16hi(y.w);
    }
}

template <int HI, bool FP8>
__global__ void __launch_bounds__(SC_THREADS, 2) score_kernel(const __grid_constant__ CUtensorMap kmap, ScoreArgs a) {
    constexpr int UB = FP8 ? SC_UNIT * 128 : SC_UNIT * 256;   // bytes per unit
    constexpr int QF4 = 8 * 8 * (HI / 2);                      // float4 entries of one warp's staged query
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* stages = smem;                                                     // SC_STAGES x 4 KiB, 1 KiB aligned
    float4* qs_all = reinterpret_cast<float4*>(smem + SC_STAGES * SC_STAGE_BYTES);  // [warp][QF4]
    float* ws_all = reinterpret_cast<float*>(qs_all + SC_CONSUMERS * QF4);        // [warp][16]
    uint64_t* full = reinterpret_cast<uint64_t*>(ws_all + SC_CONSUMERS * 16);
    uint64_t* empty = full + SC_STAGES;
    int* meta = reinterpret_cast<int*>(empty + SC_STAGES);                     // page valid flag per stage
    uint16_t* hist_all = reinterpret_cast<uint16_t*>(meta + SC_STAGES + 4);     // [warp][kHistBins], 16-bit

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();  // the top-k kernel may be scheduled now; it waits for this grid to finish
    if (a.hist)
        for (int i = threadIdx.x; i < SC_CONSUMERS * kHistBins; i += SC_THREADS) hist_all[i] = 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < SC_STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == SC_CONSUMERS) {
        // ---------------- producer warp: the 32 lanes look up the pages of 32 upcoming units
        // at once (independent loads), then lane 0 issues their TMA copies in order.
        if (lane == 0)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
        StepCursor cur;  // each lane walks the same step sequence (monotone seeks)
        bool stop = false;
        for (int64_t r = 0; !stop; ++r) {
            // unit r*32 + lane of this CTA = half (lane & 1) of this CTA's step r*16 + lane/2
            const int64_t i = r * 16 + (lane >> 1);
            const int64_t w = blockIdx.x + i * gridDim.x;
            int kind = 0;      // 0: past the end, 1: copy, 2: nothing to copy (beyond G / bad page)
            int slot = 0, page = 0;
            if (cur.seek(a, w)) {
                const int64_t gr = (w - cur.base) * SC_SUPER + (lane & 1) * SC_UNIT;
                kind = 2;
                if (gr < cur.G) {
                    const int64_t lp = gr / a.rpp;
                    slot = (int)(gr - lp * a.rpp);
                    int64_t pp = lp;
                    if (a.pt) pp = __ldg(a.pt + (int64_t)cur.b * a.pt_stride + lp);
                    if (pp >= 0 && pp < a.n_pages) {
                        kind = 1;
                        page = (int)pp;
                    } else {
                        raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                    }
                }
            }
            for (int j = 0; j < 32; ++j) {
                const int kj = __shfl_sync(0xffffffffu, kind, j);
                const int sj = __shfl_sync(0xffffffffu, slot, j);
                const int pj = __shfl_sync(0xffffffffu, page, j);
                if (kj == 0) {
                    stop = true;
                    break;
                }
                if (lane == 0) {
                    const int64_t u = r * 32 + j;  // units issued by this CTA so far
                    const int s = (int)(u % SC_STAGES);
                    if (u >= SC_STAGES && !mbar_wait(smem_u32(&empty[s]), (uint32_t)(((u / SC_STAGES) - 1) & 1))) {
                        raise_status(a.status, CSA_ERR_TIMEOUT);
                        stop = true;
                    } else {
                        const uint32_t fb = smem_u32(&full[s]);
                        if (kj == 1) {
                            meta[s] = 1;
                            mbar_arrive_expect_tx(fb, (uint32_t)UB);
                            const uint32_t dst = smem_u32(stages + s * SC_STAGE_BYTES);
                            if constexpr (FP8) {
                                tma_load_3d(dst, &kmap, 0, sj, pj, fb);
                            } else {
                                tma_load_3d(dst, &kmap, 0, sj, pj, fb);
                                tma_load_3d(dst + 2048u, &kmap, 64, sj, pj, fb);
                            }
                        } else {
                            meta[s] = 0;
                            mbar_arrive(fb);
                        }
                    }
                }
                stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
                if (stop) break;
            }
        }
        return;
    }

    // ---------------- consumers
    float4* qs = qs_all + warp * QF4;
    const uint32_t qs_addr = smem_u32(qs);
    float* wsm = ws_all + warp * 16;
    uint16_t* hist = hist_all + warp * kHistBins;
    int hist_rows = 0;  // rows counted since the last flush (16-bit counters: flush before they can wrap)
    const int r = lane & 15;        // row within its unit
    const int hu = lane >> 4;       // which of the step's two units
    int qb = -1;
    StepCursor cur;
    int64_t u = 0;
    bool waited = false;
    auto flush = [&](int req) {
        if (!waited) {  // the global histogram is cleared by the preceding kernel of the step
            pdl_wait();
            waited = true;
        }
        for (int bin = lane; bin < kHistBins; bin += 32) {
            const uint32_t c = hist[bin];
            if (c) {
                atomicAdd(a.hist + (int64_t)req * kHistBins + bin, c);
                hist[bin] = 0;
            }
        }
        hist_rows = 0;
        __syncwarp();
    };
    for (int64_t i = 0;; ++i) {
        const int64_t w = blockIdx.x + i * gridDim.x;
        if (!cur.seek(a, w)) break;
        const int64_t my_u = u;
        u += 2;
        if ((i % SC_CONSUMERS) != warp) continue;   // steps go round-robin over the consumer warps
        if (cur.b != qb) {
            if (a.hist && qb >= 0) flush(qb);
            qb = cur.b;
            // stage this request's query as {q_h[8a+i], q_h[8a+64+i]} pairs, two heads per float4
            const uint16_t* qp = a.q_idx + (int64_t)qb * a.Hi * DI;
            for (int e = lane; e < QF4; e += 32) {
                const int hp = e % (HI / 2), ii = (e / (HI / 2)) % 8, aa = e / (HI / 2) / 8;
                const int h0 = 2 * hp, h1 = 2 * hp + 1, d = 8 * aa + ii;
                float4 v;
                v.x = h0 < a.Hi ? bf16lo(qp[h0 * DI + d]) : 0.f;
                v.y = h0 < a.Hi ? bf16lo(qp[h0 * DI + d + 64]) : 0.f;
                v.z = h1 < a.Hi ? bf16lo(qp[h1 * DI + d]) : 0.f;
                v.w = h1 < a.Hi ? bf16lo(qp[h1 * DI + d + 64]) : 0.f;
                qs[e] = v;
            }
            if (lane < HI) wsm[lane] = lane < a.Hi ? __ldg(a.w_h + (int64_t)qb * a.Hi + lane) : 0.f;
            __syncwarp();
        }
        const int sA = (int)(my_u % SC_STAGES), sB = (int)((my_u + 1) % SC_STAGES);
        const bool okA = mbar_wait(smem_u32(&full[sA]), (uint32_t)((my_u / SC_STAGES) & 1));
        const bool okB = mbar_wait(smem_u32(&full[sB]), (uint32_t)(((my_u + 1) / SC_STAGES) & 1));
        if (!okA || !okB) {
            raise_status(a.status, CSA_ERR_TIMEOUT);
            break;
        }
        const int s = hu ? sB : sA;
        const int64_t g = (w - cur.base) * SC_SUPER + hu * SC_UNIT + r;
        const bool valid = g < cur.G && meta[s] != 0;
        const uint8_t* stage = stages + s * SC_STAGE_BYTES;

        float t1[HI], t2[HI], t3[HI], dot[HI];
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            const int aa = ((n & 1) << 2) | (n & 2) | ((n >> 2) & 1);  // 0,4,2,6,1,5,3,7
            float kl[8], kh[8];
            load_pair<FP8>(stage, r, aa, kl, kh);
            uint64_t acc[HI];
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const uint64_t kk = pk2(kl[ii], kh[ii]);
                const uint32_t qa = qs_addr + (uint32_t)((aa * 8 + ii) * (HI / 2)) * 16u;
#pragma unroll
                for (int hp = 0; hp < HI / 2; ++hp) {
                    uint64_t q0, q1;
                    ld_qpairs(qa + hp * 16u, q0, q1);
                    if (ii == 0) {
                        acc[2 * hp] = mul2(q0, kk);
                        acc[2 * hp + 1] = mul2(q1, kk);
                    } else {
                        acc[2 * hp] = fma2(q0, kk, acc[2 * hp]);
                        acc[2 * hp + 1] = fma2(q1, kk, acc[2 * hp + 1]);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < HI; ++h) {
                const float s1 = lo2(acc[h]) + hi2(acc[h]);       // S1[aa] = P[aa] + P[aa+8]
                if ((n & 1) == 0) {
                    t1[h] = s1;
                } else {
                    const float s2 = t1[h] + s1;                   // S2[aa-4] = S1[aa-4] + S1[aa]
                    if ((n & 3) == 1) {
                        t2[h] = s2;
                    } else {
                        const float s3 = t2[h] + s2;               // S3 = S2[t] + S2[t+2]
                        if (n == 3) t3[h] = s3;
                        else dot[h] = t3[h] + s3;                  // dot = S3[0] + S3[1]
                    }
                }
            }
        }
        // every lane has read its row: release both stages
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(smem_u32(&empty[sA]));
            mbar_arrive(smem_u32(&empty[sB]));
        }
        float sc = 0.f;
#pragma unroll
        for (int h = 0; h < HI; ++h) sc = __fmaf_rn(wsm[h], dot[h] > 0.f ? dot[h] : 0.f, sc);
        if (!valid) sc = 0.f;
        if (g < cur.G) a.scores[(int64_t)cur.b * a.score_stride + g] = sc;
        if (a.hist) {
            const bool in = g < cur.G;
            const uint32_t dg = score_key(sc) >> 21;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned peers = __match_any_sync(m, dg);
                if (lane == __ffs(peers) - 1) hist[dg] = (uint16_t)(hist[dg] + __popc(peers));  // warp-private
            }
            __syncwarp();
            hist_rows += 32;
            if (hist_rows >= 65536 - 64) flush(qb);
        }
    }
    if (a.hist && qb >= 0) flush(qb);
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// 3-D view of the index-key pool: [pages][rows per page][128 dims], box = 16 rows x
// (64 bf16 | 128 fp8) = 16 x 128 B, 128-byte swizzle.
static bool make_kmap(CUtensorMap* m, const HPaged& p, bool fp8, int64_t rows_per_page, int64_t n_pages) {
    auto enc = encoder();
    if (!enc) return false;
    const int rb = fp8 ? 128 : 256;
    cuuint64_t dims[3] = {128, (cuuint64_t)rows_per_page, (cuuint64_t)n_pages};
    cuuint64_t page_stride = p.page_stride > 0 ? (cuuint64_t)p.page_stride : (cuuint64_t)rows_per_page * rb;
    page_stride = (page_stride + 15) & ~cuuint64_t(15);
    cuuint64_t strides[2] = {(cuuint64_t)rb, page_stride};
    cuuint32_t box[3] = {fp8 ? 128u : 64u, (cuuint32_t)SC_UNIT, 1u};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void*>(p.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int HI, bool FP8>
static cudaError_t launch_score_t(const CUtensorMap& map, const ScoreArgs& a, int64_t total_steps_bound,
                                  cudaStream_t s, bool pdl) {
    constexpr int QF4 = 8 * 8 * (HI / 2);
    constexpr size_t base = 1024 + (size_t)SC_STAGES * SC_STAGE_BYTES + SC_CONSUMERS * QF4 * 16 +
                            SC_CONSUMERS * 16 * 4 + 2 * SC_STAGES * 8 + (SC_STAGES + 4) * 4;
    constexpr size_t with_hist = base + (size_t)SC_CONSUMERS * kHistBins * 2;
    const size_t smem = a.hist ? with_hist : base;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(score_kernel<HI, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)with_hist);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    }
    int64_t grid = 2LL * sms;
    if (total_steps_bound < grid) grid = total_steps_bound < 1 ? 1 : total_steps_bound;
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
    return cudaLaunchKernelEx(&cfg, score_kernel<HI, FP8>, map, a);
}

cudaError_t launch_score(const ScoreLaunch& h, cudaStream_t s, bool pdl) {
    ScoreArgs a;
    a.q_idx = static_cast<const uint16_t*>(h.q_idx);
    a.w_h = h.w_h;
    a.Hi = h.Hi;
    a.pt = h.kidx.pt;
    a.pt_stride = h.kidx.pt_stride;
    a.scores = h.scores;
    a.score_stride = h.score_stride;
    a.B = h.B;
    a.n_tokens = h.n_tokens;
    a.ratio = h.ratio;
    a.G = h.G;
    a.hist = h.hist;
    a.status = h.status;
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
    if (!make_kmap(&map, h.kidx, h.fp8, rpp, n_pages)) return cudaErrorInvalidValue;
    const int64_t steps = (int64_t)h.B * ((h.max_G + SC_SUPER - 1) / SC_SUPER);
    const int hi = h.Hi <= 4 ? 4 : (h.Hi <= 8 ? 8 : 16);
    if (h.fp8) {
        if (hi == 4) return launch_score_t<4, true>(map, a, steps, s, pdl);
        if (hi == 8) return launch_score_t<8, true>(map, a, steps, s, pdl);
        return launch_score_t<16, true>(map, a, steps, s, pdl);
    }
    if (hi == 4) return launch_score_t<4, false>(map, a, steps, s, pdl);
    if (hi == 8) return launch_score_t<8, false>(map, a, steps, s, pdl);
    return launch_score_t<16, false>(map, a, steps, s, pdl);
}

}  // namespace csa
