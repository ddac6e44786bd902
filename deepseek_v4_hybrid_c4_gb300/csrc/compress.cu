// Stage 1: softmax-gated ratio:1 compression of raw latent KV (the pages' "Flash
// Compressor": load -> gate score -> softmax -> weighted sum -> store in one
// on-chip pass; warp-local softmax for C4, one CTA per group for C128).
// ("DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "Kernel 層一堆狠活";
//  "SGLang 如何为 DeepSeek V4 打造「Day-0」推理加速", sec. "创新 2".)
//
//   s_i = x_i . w_gate + b_pos[i],  a = softmax(s),  c = sum_i a_i x_i   (fp32, bf16 out)
//
// HBM traffic is one read of the group's rows and one write of the result:
// every lane streams 32 contiguous bytes of each 1 KiB row with 16-byte loads.
#include "common.cuh"
#include "internal.h"

namespace csa {

struct CompressArgs {
    DPaged raw, out;
    const float* w_gate;
    const float* b_pos;
    const int64_t* n_tokens;
    const int64_t* n_done;
    int64_t first, count;
    int ratio;
    int nq;                    // query positions per request: histogram blocks to clear
    uint32_t* hist_zero;
    int hist_words;      // words cleared at the start of each batch entry's block
    int32_t* status;
    DWorkSet ows;              // HiSparse working set of the output pool (table == nullptr: none)
    const uint8_t* ring_pool;  // batched mode, optional: request b's token t in row
    const int32_t* ring_page;  // ring_page[b] * ring_size + t % ring_size of ring_pool
    int32_t ring_size;
    int64_t ring_n_pages;
};

__device__ __forceinline__ void group_range(const CompressArgs& a, int b, int64_t& first, int64_t& count) {
    if (a.n_tokens) {
        const int64_t G = a.n_tokens[b] / a.ratio;
        first = a.n_done[b];
        count = G - first;
        if (first < 0 || count < 0) count = 0;
    } else {
        first = a.first;
        count = a.count;
    }
}

// Raw row of token t of request b: from the compression-state ring when there is one (which
// must still hold the token: t >= n_tokens[b] - ring_size), else from the paged raw pool.
__device__ __forceinline__ const uint8_t* token_row(const CompressArgs& a, int b, int64_t t) {
    if (!a.ring_pool) return row_addr(a.raw, b, t, ROW_BYTES, a.status);
    const int64_t rp = __ldg(a.ring_page + b);
    if (rp < 0 || rp >= a.ring_n_pages || t < a.n_tokens[b] - a.ring_size) {
        raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
        return nullptr;
    }
    return a.ring_pool + (rp * a.ring_size + t % a.ring_size) * (int64_t)ROW_BYTES;
}

__device__ __forceinline__ void zero_hist(const CompressArgs& a, int b) {
    if (a.hist_zero && blockIdx.x == 0) {  // 16-byte stores: the blocks are 16-byte aligned
        const int w4 = a.hist_words / 4;
        for (int q = 0; q < a.nq; ++q) {
            uint4* z = reinterpret_cast<uint4*>(a.hist_zero + ((int64_t)b * a.nq + q) * kHistBlock);
            for (int i = threadIdx.x; i < w4; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
        }
    }
}

// lane's 16 dims of a bf16 row -> fp32
__device__ __forceinline__ void unpack16(const uint4 (&v)[2], float (&x)[16]) {
    const uint32_t w[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[2 * i] = bf16lo(w[i]);
        x[2 * i + 1] = bf16hi(w[i]);
    }
}

__device__ __forceinline__ void load_row16(const uint8_t* row, int lane, uint4 (&v)[2]) {
    if (row) {
        v[0] = ldg_nc_v4(row + lane * 32);
        v[1] = ldg_nc_v4(row + lane * 32 + 16);
    } else {
        v[0] = make_uint4(0, 0, 0, 0);
        v[1] = v[0];
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

__device__ __forceinline__ void store_row16(const DPaged& out, const DWorkSet& ws, int b, int64_t g, int lane,
                                            const float (&c)[16], int32_t* status) {
    uint8_t* dst = const_cast<uint8_t*>(row_addr(out, b, g, ROW_BYTES, status));
    if (!dst) return;
    uint8_t* dst2 = ws_slot_row(ws, out, b, g);  // the page's working-set copy, if resident
    uint4 o0, o1;
    o0.x = pack_bf16x2(c[0], c[1]);
    o0.y = pack_bf16x2(c[2], c[3]);
    o0.z = pack_bf16x2(c[4], c[5]);
    o0.w = pack_bf16x2(c[6], c[7]);
    o1.x = pack_bf16x2(c[8], c[9]);
    o1.y = pack_bf16x2(c[10], c[11]);
    o1.z = pack_bf16x2(c[12], c[13]);
    o1.w = pack_bf16x2(c[14], c[15]);
    *reinterpret_cast<uint4*>(dst + lane * 32) = o0;
    *reinterpret_cast<uint4*>(dst + lane * 32 + 16) = o1;
    if (dst2) {
        *reinterpret_cast<uint4*>(dst2 + lane * 32) = o0;
        *reinterpret_cast<uint4*>(dst2 + lane * 32 + 16) = o1;
    }
}

// C4: one warp per group of 4 tokens; gate dots reduced with warp shuffles.
__global__ void __launch_bounds__(256) compress_r4_kernel(CompressArgs a) {
    pdl_launch_dependents();  // the score kernel reads none of this kernel's outputs until its epilogue
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    zero_hist(a, b);
    int64_t first, count;
    group_range(a, b, first, count);
    float wg[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(a.w_gate + lane * 16 + i));
        wg[i] = t.x; wg[i + 1] = t.y; wg[i + 2] = t.z; wg[i + 3] = t.w;
    }
    const float bp0 = __ldg(a.b_pos + 0), bp1 = __ldg(a.b_pos + 1), bp2 = __ldg(a.b_pos + 2),
                bp3 = __ldg(a.b_pos + 3);
    const int wpb = blockDim.x >> 5;  // warps per block
    for (int64_t gi = (int64_t)blockIdx.x * wpb + warp; gi < count; gi += (int64_t)gridDim.x * wpb) {
        const int64_t g = first + gi;
        uint4 v[4][2];
#pragma unroll
        if (!a.ring_pool) {  // (uniform) the paged raw pool
#pragma unroll
            for (int i = 0; i < 4; ++i) load_row16(row_addr(a.raw, b, 4 * g + i, ROW_BYTES, a.status), lane, v[i]);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) load_row16(token_row(a, b, 4 * g + i), lane, v[i]);
        }
        float x[4][16], s[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            unpack16(v[i], x[i]);
            float p = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) p = fmaf(x[i][e], wg[e], p);
            s[i] = warp_sum(p);
        }
        s[0] += bp0; s[1] += bp1; s[2] += bp2; s[3] += bp3;
        const float m = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
        float e[4], z = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            e[i] = expf(s[i] - m);
            z += e[i];
        }
        const float inv = 1.f / z;
        float c[16];
#pragma unroll
        for (int d = 0; d < 16; ++d) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) acc = fmaf(e[i] * inv, x[i][d], acc);
            c[d] = acc;
        }
        store_row16(a.out, a.ows, b, g, lane, c, a.status);
    }
}

// C128: one CTA per group.  Warp w takes rows w, w + WARPS, ... of the group, U rows at a
// time: their page lookups go out together, then their row loads, then an online softmax over
// them (running max, sum, weighted accumulator); the WARPS partial states are merged through
// shared memory.  Decode (one pending group per request, latency-bound) runs 16 warps with all
// 8 of a warp's rows in flight; a prefill chunk (bandwidth-bound, many groups) runs 8 warps
// with 4 of 16 rows in flight, so that several CTAs share an SM.
template <int WARPS, int U>
__global__ void __launch_bounds__(WARPS * 32) compress_r128_kernel(CompressArgs a) {
    __shared__ float sm_m[WARPS], sm_l[WARPS];
    __shared__ __align__(16) float sm_acc[WARPS][D];
    pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    zero_hist(a, b);
    int64_t first, count;
    group_range(a, b, first, count);
    float wg[16];
#pragma unroll
    for (int i = 0; i < 16; i += 4) {
        const float4 t = __ldg(reinterpret_cast<const float4*>(a.w_gate + lane * 16 + i));
        wg[i] = t.x; wg[i + 1] = t.y; wg[i + 2] = t.z; wg[i + 3] = t.w;
    }
    constexpr int ROWS = 128 / WARPS;  // rows per warp
    static_assert(ROWS % U == 0, "rows per warp");
    for (int64_t gi = blockIdx.x; gi < count; gi += gridDim.x) {
        const int64_t g = first + gi;
        float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[d] = 0.f;
        for (int r0 = 0; r0 < ROWS; r0 += U) {
            const uint8_t* rows[U];
            if (!a.ring_pool) {  // (uniform) the paged raw pool: all page lookups go out together
#pragma unroll
                for (int u = 0; u < U; ++u)
                    rows[u] = row_addr(a.raw, b, 128 * g + warp + WARPS * (r0 + u), ROW_BYTES, a.status);
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) rows[u] = token_row(a, b, 128 * g + warp + WARPS * (r0 + u));
            }
            uint4 v[U][2];
#pragma unroll
            for (int u = 0; u < U; ++u) load_row16(rows[u], lane, v[u]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = warp + WARPS * (r0 + u);  // row within the group
                float x[16];
                unpack16(v[u], x);
                float p = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) p = fmaf(x[e], wg[e], p);
                const float s = warp_sum(p) + __ldg(a.b_pos + i);
                const float mn = fmaxf(m, s);
                const float sc = expf(m - mn);
                const float pe = expf(s - mn);
                l = l * sc + pe;
#pragma unroll
                for (int d = 0; d < 16; ++d) acc[d] = fmaf(pe, x[d], acc[d] * sc);
                m = mn;
            }
        }
        if (lane == 0) {
            sm_m[warp] = m;
            sm_l[warp] = l;
        }
#pragma unroll
        for (int d = 0; d < 16; d += 4)
            *reinterpret_cast<float4*>(&sm_acc[warp][lane * 16 + d]) = make_float4(acc[d], acc[d + 1], acc[d + 2], acc[d + 3]);
        __syncthreads();
        if (threadIdx.x < D / 2) {  // two columns per thread
            float M = sm_m[0];
#pragma unroll
            for (int w = 1; w < WARPS; ++w) M = fmaxf(M, sm_m[w]);
            float L = 0.f, o0 = 0.f, o1 = 0.f;
            const int d0 = 2 * threadIdx.x;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float f = expf(sm_m[w] - M);
                L = fmaf(f, sm_l[w], L);
                o0 = fmaf(f, sm_acc[w][d0], o0);
                o1 = fmaf(f, sm_acc[w][d0 + 1], o1);
            }
            const float inv = 1.f / L;
            uint8_t* dst = const_cast<uint8_t*>(row_addr(a.out, b, g, ROW_BYTES, a.status));
            const uint32_t w = pack_bf16x2(o0 * inv, o1 * inv);
            if (dst) *reinterpret_cast<uint32_t*>(dst + d0 * 2) = w;
            if (a.ows.table) {  // (uniform) the page's working-set copy, if resident
                uint8_t* dst2 = ws_slot_row(a.ows, a.out, b, g);
                if (dst && dst2) *reinterpret_cast<uint32_t*>(dst2 + d0 * 2) = w;
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- prefill chunks
// Many groups: the compression is bandwidth-bound, and per-warp row loads keep too little in
// flight (about 64 KiB per SM).  Here one thread streams the chunk's rows through a ring of
// six 32-row shared-memory stages with bulk copies (cp.async.bulk, one per run of tokens within
// a page; a group never needs a layout change), 192 KiB in flight per SM, and eight warps
// consume the stages.  C4: a stage is 8 groups, one per warp.  C128: a stage is a quarter
// group, each warp takes 4 of its rows into an online softmax carried across the quarters,
// and the 8 warps' states are merged at the group's end.  Lane l holds dims 8l .. 8l + 7 and
// 256 + 8l .. 256 + 8l + 7 of each row, so a warp's shared-memory reads are contiguous.
constexpr int CS_ROWS = 32;
constexpr int CS_STAGES = 6;
constexpr int CS_WARPS = 8;
constexpr uint32_t CS_STAGE = CS_ROWS * ROW_BYTES;
constexpr size_t CS_SMEM = (size_t)CS_STAGES * CS_STAGE + 128;

__device__ __forceinline__ void stage_row16(uint32_t row, int lane, float (&x)[16]) {
    const uint4 v[2] = {ld_shared_v4(row + (uint32_t)lane * 16u), ld_shared_v4(row + 512u + (uint32_t)lane * 16u)};
    unpack16(v, x);
}

__device__ __forceinline__ void store_row16s(const DPaged& out, int64_t g, int lane, const float (&c)[16],
                                             int32_t* status) {
    uint8_t* dst = const_cast<uint8_t*>(row_addr(out, 0, g, ROW_BYTES, status));
    if (!dst) return;
    uint4 o[2];
    uint32_t* w = reinterpret_cast<uint32_t*>(o);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(c[2 * i], c[2 * i + 1]);
    *reinterpret_cast<uint4*>(dst + lane * 16) = o[0];
    *reinterpret_cast<uint4*>(dst + 512 + lane * 16) = o[1];
}

__global__ void __launch_bounds__((CS_WARPS + 1) * 32, 1) compress_stream_kernel(CompressArgs a) {
    extern __shared__ uint8_t cs_raw[];
    __shared__ __align__(8) uint64_t full[CS_STAGES], empty[CS_STAGES];
    __shared__ float sm_m[CS_WARPS], sm_l[CS_WARPS];
    __shared__ __align__(16) float sm_acc[CS_WARPS][D];
    pdl_launch_dependents();
    const uint32_t sbase = (smem_u32(cs_raw) + 127u) & ~127u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool r4 = a.ratio == 4;
    const int64_t first = a.first, count = a.count;
    const int cpu = r4 ? 1 : 4;  // stages per unit (8 C4 groups, or one C128 group)
    const int64_t units = r4 ? (count + 7) / 8 : count;
    if (threadIdx.x == 0) {
        for (int s8 = 0; s8 < CS_STAGES; ++s8) {
            mbar_init(smem_u32(&full[s8]), 1);
            mbar_init(smem_u32(&empty[s8]), CS_WARPS);
        }
        fence_mbar_init();
    }
    __syncthreads();
    bool ok = true;
    if (warp == CS_WARPS) {  // ---- producer: one thread
        if (lane == 0) {
            const DPaged& p = a.raw;
            int64_t q = 0;
            for (int64_t u = blockIdx.x; u < units; u += gridDim.x)
                for (int c = 0; c < cpu; ++c, ++q) {
                    const int sl = (int)(q % CS_STAGES);
                    const uint32_t ph = (uint32_t)((q / CS_STAGES) & 1);
                    if (!mbar_wait(smem_u32(&empty[sl]), ph ^ 1u)) ok = false;
                    // tokens [t0, t0 + n) of this stage, in runs within a page
                    const int64_t t0 = r4 ? 4 * (first + 8 * u) : 128 * (first + u) + CS_ROWS * c;
                    const int64_t n = r4 ? 4 * (count - 8 * u < 8 ? count - 8 * u : 8) : CS_ROWS;
                    uint32_t bytes = 0;
                    for (int64_t i = 0; i < n;) {  // pass 1: the bytes that will arrive
                        const int64_t t = t0 + i, lp = t / p.rpp, run0 = p.rpp - (t - lp * p.rpp);
                        const int64_t run = run0 < n - i ? run0 : n - i;
                        const int64_t pp = p.pt ? (int64_t)__ldg(p.pt + lp) : lp;
                        if (pp >= 0 && pp < p.n_pages) bytes += (uint32_t)(run * ROW_BYTES);
                        i += run;
                    }
                    const uint32_t fb = smem_u32(&full[sl]);
                    mbar_arrive_expect_tx(fb, bytes);
                    for (int64_t i = 0; i < n;) {  // pass 2: the copies
                        const int64_t t = t0 + i, lp = t / p.rpp, sp = t - lp * p.rpp, run0 = p.rpp - sp;
                        const int64_t run = run0 < n - i ? run0 : n - i;
                        const int64_t pp = p.pt ? (int64_t)__ldg(p.pt + lp) : lp;
                        if (pp >= 0 && pp < p.n_pages)
                            bulk_g2s(sbase + (uint32_t)sl * CS_STAGE + (uint32_t)i * ROW_BYTES,
                                     p.base + pp * p.page_stride + sp * ROW_BYTES, (uint32_t)(run * ROW_BYTES), fb);
                        else
                            raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
                        i += run;
                    }
                }
            // every copy issued here is waited for by the consumers before the CTA exits
        }
    } else {  // ---- consumers
        float wg[16];
#pragma unroll
        for (int i = 0; i < 8; i += 4) {
            const float4 t0 = __ldg(reinterpret_cast<const float4*>(a.w_gate + lane * 8 + i));
            const float4 t1 = __ldg(reinterpret_cast<const float4*>(a.w_gate + 256 + lane * 8 + i));
            wg[i] = t0.x; wg[i + 1] = t0.y; wg[i + 2] = t0.z; wg[i + 3] = t0.w;
            wg[8 + i] = t1.x; wg[8 + i + 1] = t1.y; wg[8 + i + 2] = t1.z; wg[8 + i + 3] = t1.w;
        }
        int64_t q = 0;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
            float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
            for (int d = 0; d < 16; ++d) acc[d] = 0.f;
            for (int c = 0; c < cpu; ++c, ++q) {
                const int sl = (int)(q % CS_STAGES);
                const uint32_t ph = (uint32_t)((q / CS_STAGES) & 1);
                if (!mbar_wait(smem_u32(&full[sl]), ph)) ok = false;
                const uint32_t st = sbase + (uint32_t)sl * CS_STAGE + (uint32_t)warp * 4u * ROW_BYTES;
                if (r4) {
                    const int64_t gi = 8 * u + warp;
                    if (gi < count) {
                        float x[4][16], s[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            stage_row16(st + (uint32_t)i * ROW_BYTES, lane, x[i]);
                            float pd = 0.f;
#pragma unroll
                            for (int e = 0; e < 16; ++e) pd = fmaf(x[i][e], wg[e], pd);
                            s[i] = warp_sum(pd) + __ldg(a.b_pos + i);
                        }
                        const float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
                        float e[4], z = 0.f;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            e[i] = expf(s[i] - mx);
                            z += e[i];
                        }
                        const float inv = 1.f / z;
                        float cc[16];
#pragma unroll
                        for (int d = 0; d < 16; ++d) {
                            float t = 0.f;
#pragma unroll
                            for (int i = 0; i < 4; ++i) t = fmaf(e[i] * inv, x[i][d], t);
                            cc[d] = t;
                        }
                        store_row16s(a.out, first + gi, lane, cc, a.status);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        float x[16];
                        stage_row16(st + (uint32_t)i * ROW_BYTES, lane, x);
                        float pd = 0.f;
#pragma unroll
                        for (int e = 0; e < 16; ++e) pd = fmaf(x[e], wg[e], pd);
                        const float sv = warp_sum(pd) + __ldg(a.b_pos + CS_ROWS * c + 4 * warp + i);
                        const float mn = fmaxf(m, sv);
                        const float sc = expf(m - mn);
                        const float pe = expf(sv - mn);
                        l = l * sc + pe;
#pragma unroll
                        for (int d = 0; d < 16; ++d) acc[d] = fmaf(pe, x[d], acc[d] * sc);
                        m = mn;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[sl]));
            }
            if (!r4) {  // merge the 8 warps' states: thread t finishes columns 2t, 2t + 1
                if (lane == 0) {
                    sm_m[warp] = m;
                    sm_l[warp] = l;
                }
#pragma unroll
                for (int d = 0; d < 8; ++d) {
                    sm_acc[warp][lane * 8 + d] = acc[d];
                    sm_acc[warp][256 + lane * 8 + d] = acc[8 + d];
                }
                named_bar_sync(1, CS_WARPS * 32);
                float M = sm_m[0];
#pragma unroll
                for (int w = 1; w < CS_WARPS; ++w) M = fmaxf(M, sm_m[w]);
                float L = 0.f, o0 = 0.f, o1 = 0.f;
                const int d0 = 2 * threadIdx.x;
#pragma unroll
                for (int w = 0; w < CS_WARPS; ++w) {
                    const float f = expf(sm_m[w] - M);
                    L = fmaf(f, sm_l[w], L);
                    o0 = fmaf(f, sm_acc[w][d0], o0);
                    o1 = fmaf(f, sm_acc[w][d0 + 1], o1);
                }
                const float inv = 1.f / L;
                uint8_t* dst = const_cast<uint8_t*>(row_addr(a.out, 0, first + u, ROW_BYTES, a.status));
                if (dst) *reinterpret_cast<uint32_t*>(dst + d0 * 2) = pack_bf16x2(o0 * inv, o1 * inv);
                named_bar_sync(1, CS_WARPS * 32);
            }
        }
    }
    if (!ok) raise_status(a.status, CSA_ERR_TIMEOUT);
}

static DPaged to_dev(const HPaged& h) {
    DPaged d;
    d.base = static_cast<const uint8_t*>(h.base);
    d.pt = h.pt;
    d.pt_stride = h.pt_stride;
    d.page_stride = h.page_stride;
    d.n_pages = h.n_pages;
    d.rpp = h.rpp;
    d.qpr = h.qpr > 1 ? h.qpr : 1;
    return d;
}

cudaError_t launch_compress(const CompressLaunch& h, cudaStream_t s, bool pdl) {
    CompressArgs a;
    a.raw = to_dev(h.raw);
    a.out = to_dev(h.out);
    a.w_gate = h.w_gate;
    a.b_pos = h.b_pos;
    a.n_tokens = h.n_tokens;
    a.n_done = h.n_done;
    a.first = h.first;
    a.count = h.count;
    a.ratio = h.ratio;
    a.hist_zero = h.hist_zero;
    a.hist_words = h.hist_words > 0 && h.hist_words <= kHistBlock ? h.hist_words : kHistBlock;
    a.nq = h.nq > 1 ? h.nq : 1;
    a.status = h.status;
    a.ring_pool = h.n_tokens ? static_cast<const uint8_t*>(h.ring_pool) : nullptr;  // batched mode only
    a.ows.table = h.n_tokens ? h.hs.table : nullptr;
    a.ows.base = static_cast<uint8_t*>(h.hs.base);
    a.ows.n_slots = h.hs.n_slots;
    a.ows.touch = nullptr;
    a.ows.step = 0;
    a.ring_page = h.ring_page;
    a.ring_size = h.ring_size;
    a.ring_n_pages = h.ring_n_pages;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.stream = s;
    const int sms = device_sm_count();
    if (!sms) return cudaErrorInvalidDevice;
    if (!h.n_tokens && h.B == 1 && (h.ratio == 4 ? (h.count + 7) / 8 : h.count) >= sms) {
        // a prefill chunk that fills every SM: stream it through shared memory
        cudaError_t e = set_func_attr_once((const void*)compress_stream_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)CS_SMEM);
        if (e != cudaSuccess) return e;
        cfg.blockDim = dim3((CS_WARPS + 1) * 32, 1, 1);
        cfg.gridDim = dim3((unsigned)sms, 1, 1);
        cfg.dynamicSmemBytes = CS_SMEM;
        return cudaLaunchKernelEx(&cfg, compress_stream_kernel, a);
    }
    // C128: a few groups (decode, a short chunk) are latency-bound, many are bandwidth-bound
    const bool r128_wide = h.n_tokens != nullptr || h.count < 152;
    cfg.blockDim = dim3(h.ratio == 4 ? 256 : (r128_wide ? 16 : 8) * 32, 1, 1);
    int64_t gx;
    if (h.n_tokens) {
        gx = 1;  // decode: one block per request loops over its pending groups
        // C4: a single warp, small enough to share an SM with the index-score kernel's CTAs
        // (which start right behind it and fill every SM)
        if (h.ratio == 4) cfg.blockDim = dim3(32, 1, 1);
    } else {
        gx = h.ratio == 4 ? (h.count + 7) / 8 : h.count;
    }
    if (gx < 1) gx = 1;
    if (gx > 0x7FFFFFFFLL) gx = 0x7FFFFFFFLL;
    cfg.gridDim = dim3((unsigned)gx, (unsigned)h.B, 1);
    if (h.ratio == 4) {
        // the carveout the caller asks for: the SM that runs this warp then keeps room for the
        // score kernel's CTAs, which start right behind it (a CTA can join an SM only in the
        // shared-memory configuration the SM runs in)
        cudaError_t e = set_func_attr_once((const void*)compress_r4_kernel,
                                           cudaFuncAttributePreferredSharedMemoryCarveout, h.carveout);
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, compress_r4_kernel, a);
    }
    return r128_wide ? cudaLaunchKernelEx(&cfg, compress_r128_kernel<16, 8>, a)
                     : cudaLaunchKernelEx(&cfg, compress_r128_kernel<8, 4>, a);
}

}  // namespace csa
