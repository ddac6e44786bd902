// Stage 2: indexer score of every compressed candidate ("DeepSeek-V4 本地部署，SGLang
// 把活做絕了", sec. "Kernel 層一堆狠活": 256K candidates at 1M context feed the top-512).
//
//   score[g] = sum_h w_h * ReLU(q_idx[h] . k_idx[g])     fp32, bit-exact fixed order:
//   Q[j]  = q[32j]*k[32j], then fma over dims 32j+1..32j+31   (chain j = 0..3)
//   dot   = (Q[0] + Q[2]) + (Q[1] + Q[3])
//   acc   = fma(w_h, ReLU(dot_h), acc) for h = 0..Hi-1, from acc = 0
//
// Layout: a warp takes a step of 32 rows (two 16-row units).  Lane (c, r), c = lane / 16,
// r = lane % 16, holds rows r and r+16 and runs chains c and c+2 of both rows together with
// packed fma.rn.f32x2 (the two halves of a 64-bit accumulator are the Q[c] and Q[c+2]
// chains -- two IEEE fmas per instruction, dims 32c+i and 64+32c+i).  Half c ends with
// Q[c] + Q[c+2]; one shuffle across the halves gives the dot (IEEE addition is
// commutative, so both halves agree bit for bit), and lane l finishes row l.  The index
// query is staged in shared memory as {q[32c+i], q[64+32c+i]} pairs, two heads per
// 16-byte load, and each load feeds both of the lane's rows.
//
// Memory path: each warp owns two 32-row slots in shared memory and fills them with TMA
// tensor copies (cp.async.bulk.tensor, 128-byte swizzle), two units per step, completing
// on the slot's mbarrier; it refills a slot as soon as every lane has read it, so a step
// is always in flight behind the one being computed.  Page-table lookups are batched 16
// steps ahead.  The swizzle puts 16-byte chunk c of row r at position c ^ (r & 7), so the
// lanes' reads of one logical chunk of 16 rows spread over the banks.
//
// Scheduling: one CTA per SM, one wave: 12 warps (6 for 16 index heads).  Two CTAs of 6 warps
// per SM ran unevenly: the warp schedulers favour older warps, so the CTA dispatched first to an
// SM finished well before its partner (by half on the fp8 path), which then ran alone.  The work
// is cut into CTA-steps of W consecutive steps of one request (warp j takes step j), so all warps
// of a CTA work on the same request at a time and share one staged query and one histogram.
// With one batch entry every CTA takes an equal contiguous range of steps.
//
// Optional fused epilogue: a per-CTA histogram of the top 11 bits of each score's
// order-preserving key (the first digit of the top-k radix select), flushed per
// request into a global [B][2048] histogram.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace csa {

// Warps per CTA (one CTA per SM); each takes 32 rows (2 units) per CTA-step.  Up to 8 index heads
// twelve warps fit the register file (capped at 160 registers per thread: same box, 1M step 41.51
// against 41.75 us at 162); 16 heads need more registers per thread and run six.
template <int HI>
__host__ __device__ constexpr int sc_warps() { return HI >= 16 ? 6 : 12; }
constexpr int SC_UNIT = 16;                  // rows per unit (one TMA box height)
constexpr int SC_SUPER = 32;                 // rows per warp step
constexpr int SC_STAGE_BYTES = SC_UNIT * 256;  // one unit (bf16; fp8 uses half)
constexpr int SC_SLOT_BYTES = 2 * SC_STAGE_BYTES;  // one step

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
    int nq;                  // query positions per request (batch entry b: request b / nq)
    int64_t G;
    uint32_t* hist;          // [B][kHistBlock] (the first kHistBins words) or nullptr
    int32_t* status;
};
// With one batch entry, CTA i of n takes the steps [i S / n, (i + 1) S / n) of the S = ceil(G / 32)
// 32-row steps: its CTA-step k covers steps s0 + W k .. s0 + W k + W - 1 (warp j the j-th), clipped
// at s1.

// Walks the concatenated CTA-steps of the batch.  Request b has steps = ceil(G_b / 32)
// steps of 32 rows, grouped into ceil(steps / W) CTA-steps of W consecutive steps (warp j of
// the CTA takes step j), so a CTA-step never straddles two requests.  After seek(m), CTA-step m
// belongs to request b.  Calls must come with non-decreasing m.
template <int W>
struct CtaStepCursor {
    int b = -1;
    int64_t base = 0, csteps = 0, steps = 0, G = 0;
    __device__ void load(const ScoreArgs& a) {
        G = a.n_tokens ? query_tokens(a.n_tokens, b, a.nq) / a.ratio : a.G;
        steps = (G + SC_SUPER - 1) / SC_SUPER;
        csteps = (steps + W - 1) / W;
    }
    // Start at request b0, whose first CTA-step is base0 (every later seek must lie at or past it).
    __device__ void start(const ScoreArgs& a, int b0, int64_t base0) {
        b = b0 < a.B ? b0 : a.B;
        base = base0;
        if (b < a.B) load(a);
    }
    __device__ bool seek(const ScoreArgs& a, int64_t m) {
        if (b < 0) {
            if (a.B <= 0) return false;
            b = 0;
            load(a);
        }
        if (b >= a.B) return false;  // stays past the end once there
        while (m >= base + csteps) {
            base += csteps;
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

// Several batch entries: this CTA's contiguous share [m0, m0 + nk) of the batch's CTA-steps,
// the request holding CTA-step m0 (b_start) and that request's first CTA-step (base_start).
template <int SC_WARPS>
__device__ __forceinline__ void batch_share(const ScoreArgs& a, int64_t& m0, int64_t& nk, int& b_start,
                                         int64_t& base_start) {
    constexpr int SC_THREADS = SC_WARPS * 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ int64_t s_tot[SC_WARPS];
    int64_t t = 0;  // the batch's CTA-steps (ragged requests: from the device lengths)
    for (int b = threadIdx.x; b < a.B; b += SC_THREADS) {
        const int64_t G = a.n_tokens ? query_tokens(a.n_tokens, b, a.nq) / a.ratio : a.G;
        t += ((G + SC_SUPER - 1) / SC_SUPER + SC_WARPS - 1) / SC_WARPS;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) s_tot[warp] = t;
    __syncthreads();
    int64_t total = 0;
#pragma unroll
    for (int w = 0; w < SC_WARPS; ++w) total += s_tot[w];
    m0 = (int64_t)blockIdx.x * total / gridDim.x;
    nk = ((int64_t)blockIdx.x + 1) * total / gridDim.x - m0;
    // The request holding CTA-step m0 and its first CTA-step, by a prefix over the requests in
    // chunks of SC_THREADS: the cursors start there.  (Walking from request 0 costs one
    // dependent length load per request: about 17 us before the first copy for a CTA that
    // starts 25 requests into a 32-request batch.)
    __shared__ int s_b0;
    __shared__ int64_t s_base0, s_part[SC_WARPS];
    if (threadIdx.x == 0) {
        s_b0 = a.B;
        s_base0 = total;
    }
    int64_t carry = 0;
    for (int c0 = 0; c0 < a.B; c0 += SC_THREADS) {
        const int b = c0 + (int)threadIdx.x;
        int64_t cs = 0;
        if (b < a.B) {
            const int64_t G = a.n_tokens ? query_tokens(a.n_tokens, b, a.nq) / a.ratio : a.G;
            cs = ((G + SC_SUPER - 1) / SC_SUPER + SC_WARPS - 1) / SC_WARPS;
        }
        int64_t x = cs;  // inclusive prefix within the warp
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __syncthreads();  // (s_part's previous chunk read, s_b0 written)
        if (lane == 31) s_part[warp] = x;
        __syncthreads();
        int64_t before = 0, chunk = 0;
        for (int w = 0; w < SC_WARPS; ++w) {
            before += w < warp ? s_part[w] : 0;
            chunk += s_part[w];
        }
        const int64_t first = carry + before + x - cs;  // request b's first CTA-step
        if (b < a.B && cs > 0 && m0 >= first && m0 < first + cs) {
            s_b0 = b;
            s_base0 = first;
        }
        carry += chunk;
        __syncthreads();
        if (s_b0 < a.B) break;  // (the same for every thread)
    }
    b_start = s_b0;
    base_start = s_base0;
}

// BLK: several batch entries (contiguous shares of the batch's CTA-steps); otherwise one entry.
// The two are separate instantiations: with the several-entry set-up compiled into the one-entry
// kernel, the 1M step measured 0.8-1.8 us slower (same box).
template <int HI, bool FP8, bool BLK>
__global__ void __launch_bounds__(sc_warps<HI>() * 32) __maxnreg__(HI >= 16 ? 255 : 160)
    score_kernel(const __grid_constant__ CUtensorMap kmap, ScoreArgs a) {
    constexpr int SC_WARPS = sc_warps<HI>(), SC_THREADS = SC_WARPS * 32;
    constexpr int UB = FP8 ? SC_UNIT * 128 : SC_UNIT * 256;   // bytes per 16-row unit
    constexpr int QF4 = 32 * (HI / 2) * 2;                     // float4 entries of the staged query
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // per warp: two 32-row slots; per CTA: the staged query, the weights, the histogram
    uint8_t* slots = smem + warp * (2 * SC_SLOT_BYTES);
    float4* qs = reinterpret_cast<float4*>(smem + SC_WARPS * 2 * SC_SLOT_BYTES);
    float* wsm = reinterpret_cast<float*>(smem + SC_WARPS * 2 * SC_SLOT_BYTES + QF4 * 16);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + SC_WARPS * 2 * SC_SLOT_BYTES + QF4 * 16 + 64) + warp * 2;
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + SC_WARPS * 2 * SC_SLOT_BYTES + QF4 * 16 + 64 +
                                                 SC_WARPS * 16);
    const uint32_t qs_addr = smem_u32(qs);

    pdl_launch_dependents();  // the top-k kernel may be scheduled now; it waits for this grid to finish
    if (a.hist)
        for (int i = threadIdx.x; i < kHistBins; i += SC_THREADS) hist[i] = 0;
    if (lane == 0) {
        mbar_init(smem_u32(&full[0]), 2);
        mbar_init(smem_u32(&full[1]), 2);
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
    }
    __syncwarp();

    // This CTA's CTA-steps: one request -- m = blockIdx.x + k gridDim.x, k = 0, 1, ...; a batch
    // -- a contiguous share [m0, m0 + nk) of its CTA-steps, so that a CTA meets one or two
    // requests rather than a new one (query restage, histogram flush) every CTA-step.  In each
    // CTA-step warp j takes step j.  Page lookups run a window of 16 CTA-steps at a time: lane l
    // holds unit
    // (l & 1) of this warp's step in CTA-step k0 + (l >> 1), all 32 loads in flight together.
    // Two register sets alternate (even / odd windows) and the next window is looked up as the
    // current one starts, so the page-table latency stays off the copy path.
    constexpr bool blocked = BLK;
    int64_t m0 = blockIdx.x, nk = INT64_MAX;
    int b_start = 0;          // the cursors' starting request and its first CTA-step
    int64_t base_start = 0;
    int64_t s0 = 0, s1 = 0;  // one batch entry: this CTA's steps [s0, s1)
    if (!blocked) {
        const int64_t G0 = a.B < 1 ? 0 : (a.n_tokens ? query_tokens(a.n_tokens, 0, a.nq) / a.ratio : a.G);
        const int64_t S0 = (G0 + SC_SUPER - 1) / SC_SUPER;
        s0 = (int64_t)blockIdx.x * S0 / gridDim.x;
        s1 = ((int64_t)blockIdx.x + 1) * S0 / gridDim.x;
        nk = (s1 - s0 + SC_WARPS - 1) / SC_WARPS;
    } else {
        if constexpr (BLK) batch_share<SC_WARPS>(a, m0, nk, b_start, base_start);
    }
    // the CTA-step index of the CTA's k-th CTA-step (one batch entry: 0, the entry's; the warp's
    // step then comes from s0), and warp `warp`'s step within its request, or -1 past the CTA's range
    auto cta_step = [&](int64_t k) { return blocked ? m0 + k : (int64_t)0; };
    auto warp_step = [&](int64_t k, int64_t m, int64_t base) -> int64_t {
        if (blocked) return (m - base) * SC_WARPS + warp;
        const int64_t st = s0 + k * SC_WARPS + warp;
        return st < s1 ? st : -1;
    };
    CtaStepCursor<SC_WARPS> lc;  // this lane's lookup cursor
    if constexpr (BLK) lc.start(a, b_start, base_start);
    int wk[2] = {0, 0}, ws[2] = {0, 0}, wp[2] = {0, 0};  // per set: kind (0 past the end, 1 copy,
                                                          // 2 nothing to copy), row in page, page
    auto lookup_window = [&](int64_t k0, int& kind, int& slot, int& page) {
        const int64_t k = k0 + (lane >> 1);
        kind = 0;
        slot = 0;
        page = 0;
        const int64_t m = cta_step(k);
        if (k < nk && lc.seek(a, m)) {
            const int64_t ws_ = warp_step(k, m, lc.base);
            const int64_t gr = ws_ * SC_SUPER + (lane & 1) * SC_UNIT;
            kind = 2;
            if (ws_ >= 0 && gr < lc.G) {
                const int64_t lp = gr / a.rpp;
                slot = (int)(gr - lp * a.rpp);
                int64_t pp = lp;
                if (a.pt) pp = __ldg(a.pt + (int64_t)(a.nq > 1 ? lc.b / a.nq : lc.b) * a.pt_stride + lp);
                if (pp >= 0 && pp < a.n_pages) {
                    kind = 1;
                    page = (int)pp;
                } else {
                    raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                }
            }
        }
    };
    // Fetch this warp's step of CTA-step k into slot k & 1: lanes 2i, 2i+1 (i = k mod 16) hold
    // its two units.
    auto issue = [&](int64_t k) {
        const int set = (int)((k >> 4) & 1);
        const int kind = set ? wk[1] : wk[0];
        if ((lane >> 1) == (int)(k & 15) && kind != 0) {
            const int sl = (int)(k & 1);
            const uint32_t fb = smem_u32(&full[sl]);
            if (kind == 1) {
                const int slot = set ? ws[1] : ws[0], page = set ? wp[1] : wp[0];
                mbar_arrive_expect_tx(fb, (uint32_t)UB);
                const uint32_t dst = smem_u32(slots + sl * SC_SLOT_BYTES + (lane & 1) * SC_STAGE_BYTES);
                if constexpr (FP8) {
                    tma_load_3d(dst, &kmap, 0, slot, page, fb);
                } else {
                    tma_load_3d(dst, &kmap, 0, slot, page, fb);
                    tma_load_3d(dst + 2048u, &kmap, 64, slot, page, fb);
                }
            } else {
                mbar_arrive(fb);
            }
        }
    };
    // The index query of a request: thread t holds 16-byte chunks t and t + SC_THREADS of the
    // [Hi][128] bf16 rows (chunk j = head j / 16, dims 8 (j % 16) ..), and thread t < HI the
    // head weight.  A request's query is fetched one CTA-step before it is staged, so its
    // loads never queue behind the bulk copies; the first one is fetched before any copy.
    constexpr int QCH = HI * DI / 8;  // 16-byte chunks of the query, HI <= 16 -> <= 256
    uint4 qv[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    float wv = 0.f;
    int qf_b = -1;  // request whose query the registers hold (CTA-uniform)
    auto q_fetch = [&](int b) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q_idx + (int64_t)b * a.Hi * DI);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int j = threadIdx.x + i * SC_THREADS;
            qv[i] = (j < QCH && j / 16 < a.Hi) ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
        }
        wv = threadIdx.x < a.Hi ? __ldg(a.w_h + (int64_t)b * a.Hi + threadIdx.x) : 0.f;
        qf_b = b;
    };
    // Staged layout: float4 (i * HI/2 + head pair) * 2 + c holds {q_h0[32c+i], q_h0[64+32c+i],
    // q_h1[32c+i], q_h1[64+32c+i]}, i = 0..31.
    auto q_store = [&]() {
        float* qf = reinterpret_cast<float*>(qs);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int j = threadIdx.x + i * SC_THREADS;
            if (j < QCH) {
                const int h = j >> 4, d0 = (j & 15) * 8;
                const uint32_t wd[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int d = d0 + e, dd = d & 63;
                    const int idx = (((dd & 31) * (HI / 2) + (h >> 1)) * 2 + (dd >> 5)) * 4 + (h & 1) * 2 + (d >> 6);
                    qf[idx] = (e & 1) ? bf16hi(wd[e >> 1]) : bf16lo(wd[e >> 1]);
                }
            }
        }
        if (threadIdx.x < HI) wsm[threadIdx.x] = wv;
    };
    {
        CtaStepCursor<SC_WARPS> c0;
        if constexpr (BLK) c0.start(a, b_start, base_start);
        if (nk > 0 && c0.seek(a, cta_step(0))) q_fetch(c0.b);
    }
    lookup_window(0, wk[0], ws[0], wp[0]);
    lookup_window(16, wk[1], ws[1], wp[1]);
    issue(0);
    issue(1);

    int qb = -1;
    bool dead = false;    // a copy never arrived: stop waiting and fetching, keep the CTA barriers
    bool waited = false;
    auto flush = [&](int req) {  // whole CTA
        if (!waited) {  // the global histogram is cleared by the preceding kernel of the step
            pdl_wait();
            waited = true;
        }
        for (int bin = threadIdx.x; bin < kHistBins; bin += SC_THREADS) {
            const uint32_t c = hist[bin];
            if (c) {
                atomicAdd(a.hist + (int64_t)req * kHistBlock + bin, c);
                hist[bin] = 0;
            }
        }
    };
    const int r = lane & 15;        // row within its unit
    const int hu = lane >> 4;       // chunk half (c)
    CtaStepCursor<SC_WARPS> cur;
    if constexpr (BLK) cur.start(a, b_start, base_start);
    for (int64_t k = 0;; ++k) {
        const int64_t m = cta_step(k);
        if (k >= nk || !cur.seek(a, m)) break;  // the same for every warp of the CTA
        const int sl = (int)(k & 1);
        if ((k & 15) == 0 && k > 0) {  // window k/16 starts: look up window k/16 + 1 into the freed set
            if ((k >> 4) & 1) lookup_window(k + 16, wk[0], ws[0], wp[0]);
            else lookup_window(k + 16, wk[1], ws[1], wp[1]);
        }
        if (cur.b != qb) {  // CTA-uniform: restage the query, flush the previous request's histogram
            if (qf_b != cur.b) q_fetch(cur.b);
            __syncthreads();
            if (a.hist && qb >= 0) flush(qb);
            qb = cur.b;
            q_store();
            __syncthreads();
        }
        {  // the CTA's next CTA-step starts another request: fetch its query now
            CtaStepCursor<SC_WARPS> nx = cur;
            if (k + 1 < nk && nx.seek(a, cta_step(k + 1)) && nx.b != qb && nx.b != qf_b) q_fetch(nx.b);
        }
        const int64_t st = warp_step(k, m, cur.base);  // this warp's step within the request (-1: none)
        const int kind_me = __shfl_sync(0xffffffffu, ((k >> 4) & 1) ? wk[1] : wk[0], 2 * (int)(k & 15) + hu);
        if (!dead && !mbar_wait(smem_u32(&full[sl]), (uint32_t)((k >> 1) & 1))) {
            raise_status(a.status, CSA_ERR_TIMEOUT);
            dead = true;
        }
        if (dead) continue;
        if (st < 0 || st >= cur.steps) {  // the request's (or this CTA's) last CTA-step has fewer steps than warps
            issue(k + 2);
            continue;
        }
        const int64_t g = st * SC_SUPER + lane;
        const bool valid = g < cur.G && kind_me == 1;
        // lane (c, r): rows r and r+16 of the step (units 0 and 1, in-unit row r); chains c
        // and c+2: dims 32c + 8g + ii (low halves) and 64 + 32c + 8g + ii (high halves)
        const uint8_t* st0 = slots + sl * SC_SLOT_BYTES;
        const uint8_t* st1 = st0 + SC_STAGE_BYTES;
        uint64_t acc0[HI], acc1[HI];
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) {
            const int ch = 4 * hu + gq;  // 8-dim chunk of each half row
            float kl0[8], kh0[8], kl1[8], kh1[8];
            load_pair<FP8>(st0, r, ch, kl0, kh0);
            load_pair<FP8>(st1, r, ch, kl1, kh1);
#pragma unroll
            for (int ii = 0; ii < 8; ++ii) {
                const uint64_t kk0 = pk2(kl0[ii], kh0[ii]);
                const uint64_t kk1 = pk2(kl1[ii], kh1[ii]);
                const uint32_t qa = qs_addr + (uint32_t)(((gq * 8 + ii) * (HI / 2)) * 2 + hu) * 16u;
#pragma unroll
                for (int hp = 0; hp < HI / 2; ++hp) {
                    uint64_t q0, q1;
                    ld_qpairs(qa + hp * 32u, q0, q1);
                    // each pair of consecutive instructions shares one multiplicand
                    if (gq == 0 && ii == 0) {
                        acc0[2 * hp] = mul2(q0, kk0);
                        acc1[2 * hp] = mul2(q0, kk1);
                        acc1[2 * hp + 1] = mul2(q1, kk1);
                        acc0[2 * hp + 1] = mul2(q1, kk0);
                    } else {
                        acc0[2 * hp] = fma2(q0, kk0, acc0[2 * hp]);
                        acc1[2 * hp] = fma2(q0, kk1, acc1[2 * hp]);
                        acc1[2 * hp + 1] = fma2(q1, kk1, acc1[2 * hp + 1]);
                        acc0[2 * hp + 1] = fma2(q1, kk0, acc0[2 * hp + 1]);
                    }
                }
            }
        }
        // every lane has read the slot: refill it with the CTA-step after next
        __syncwarp();
        issue(k + 2);
        float dot[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) {
            const float r0 = lo2(acc0[h]) + hi2(acc0[h]);  // row r:    Q[c] + Q[c+2]
            const float r1 = lo2(acc1[h]) + hi2(acc1[h]);  // row r+16
            const float other = __shfl_xor_sync(0xffffffffu, hu ? r0 : r1, 16);
            dot[h] = (hu ? r1 : r0) + other;               // (Q[0] + Q[2]) + (Q[1] + Q[3])
        }
        float sc = 0.f;
#pragma unroll
        for (int h = 0; h < HI; ++h) sc = __fmaf_rn(wsm[h], dot[h] > 0.f ? dot[h] : 0.f, sc);
        if (!valid) sc = 0.f;
        if (g < cur.G) a.scores[(int64_t)cur.b * a.score_stride + g] = sc;
        if (a.hist) {
            const bool in = g < cur.G;
            const uint32_t dg = score_key(sc) >> 21;
            const unsigned mk = __ballot_sync(0xffffffffu, in);
            if (in) {
                const unsigned peers = __match_any_sync(mk, dg);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[dg], (uint32_t)__popc(peers));
            }
        }
    }
    __syncthreads();
    if (a.hist && qb >= 0) flush(qb);
    // Nothing is in flight here on a normal exit: the two CTA-steps looked up last lie past
    // the end, so no copy was issued for them.
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
bool make_kidx_map(void* map, const HPaged& p, bool fp8, int64_t rows_per_page, int64_t n_pages) {
    CUtensorMap* m = static_cast<CUtensorMap*>(map);
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

template <int HI, bool FP8, bool BLK>
static cudaError_t launch_score_t(const CUtensorMap& map, const ScoreArgs& a, int64_t max_steps,
                                  int reserve, cudaStream_t s, bool pdl) {
    constexpr int QF4 = 8 * 8 * (HI / 2);
    constexpr int SC_WARPS = sc_warps<HI>();
    constexpr size_t base = 1024 + (size_t)SC_WARPS * 2 * SC_SLOT_BYTES + (size_t)QF4 * 16 + 64 + SC_WARPS * 16;
    constexpr size_t with_hist = base + (size_t)kHistBins * 4;
    const size_t smem = a.hist ? with_hist : base;
    {
        cudaError_t e = set_func_attr_once((const void*)score_kernel<HI, FP8, BLK>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)with_hist);
        if (e != cudaSuccess) return e;
    }
    const int sms = device_sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    int64_t grid = (int64_t)sms - reserve;  // one wave: a CTA per SM
    const int64_t total_steps_bound = (int64_t)a.B * ((max_steps + SC_WARPS - 1) / SC_WARPS);
    if (grid < 1) grid = 1;
    if (total_steps_bound < grid) grid = total_steps_bound < 1 ? 1 : total_steps_bound;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(SC_WARPS * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, score_kernel<HI, FP8, BLK>, map, a);
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
    a.nq = h.nq > 1 ? h.nq : 1;
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
    if (!make_kidx_map(&map, h.kidx, h.fp8, rpp, n_pages)) return cudaErrorInvalidValue;
    const int64_t steps = (h.max_G + SC_SUPER - 1) / SC_SUPER;  // 32-row steps of the longest request
    const int hi = h.Hi <= 4 ? 4 : (h.Hi <= 8 ? 8 : 16);
    const bool blk = h.B > 1;
    auto go = [&](auto fp8, auto blkc) -> cudaError_t {
        constexpr bool F = decltype(fp8)::value, K = decltype(blkc)::value;
        if (hi == 4) return launch_score_t<4, F, K>(map, a, steps, h.reserve, s, pdl);
        if (hi == 8) return launch_score_t<8, F, K>(map, a, steps, h.reserve, s, pdl);
        return launch_score_t<16, F, K>(map, a, steps, h.reserve, s, pdl);
    };
    using T = std::true_type;
    using F = std::false_type;
    if (h.fp8) return blk ? go(T{}, T{}) : go(T{}, F{});
    return blk ? go(F{}, T{}) : go(F{}, F{});
}

}  // namespace csa
