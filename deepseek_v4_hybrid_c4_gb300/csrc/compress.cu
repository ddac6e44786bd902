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
    uint32_t* hist_zero;
    int32_t* status;
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

__device__ __forceinline__ void zero_hist(const CompressArgs& a, int b) {
    if (a.hist_zero && blockIdx.x == 0) {  // 16-byte stores: the block is 16-byte aligned
        uint4* z = reinterpret_cast<uint4*>(a.hist_zero + (int64_t)b * kHistBlock);
        for (int i = threadIdx.x; i < kHistBlock / 4; i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
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

__device__ __forceinline__ void store_row16(const DPaged& out, int b, int64_t g, int lane, const float (&c)[16],
                                            int32_t* status) {
    uint8_t* dst = const_cast<uint8_t*>(row_addr(out, b, g, ROW_BYTES, status));
    if (!dst) return;
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
        for (int i = 0; i < 4; ++i) load_row16(row_addr(a.raw, b, 4 * g + i, ROW_BYTES, a.status), lane, v[i]);
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
        store_row16(a.out, b, g, lane, c, a.status);
    }
}

// C128: one CTA (16 warps) per group.  Warp w takes rows w, w + 16, ..., w + 112 of the
// group: their page lookups go out together, then all 8 row loads, then an online softmax
// over the 8 rows (running max, sum, weighted accumulator); the 16 partial states are merged
// through shared memory.
constexpr int R128_WARPS = 16;
__global__ void __launch_bounds__(R128_WARPS * 32) compress_r128_kernel(CompressArgs a) {
    __shared__ float sm_m[R128_WARPS], sm_l[R128_WARPS];
    __shared__ __align__(16) float sm_acc[R128_WARPS][D];
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
    constexpr int ROWS = 128 / R128_WARPS;  // 8 rows per warp, all in flight
    for (int64_t gi = blockIdx.x; gi < count; gi += gridDim.x) {
        const int64_t g = first + gi;
        const uint8_t* rows[ROWS];
#pragma unroll
        for (int u = 0; u < ROWS; ++u) rows[u] = row_addr(a.raw, b, 128 * g + warp + R128_WARPS * u, ROW_BYTES, a.status);
        uint4 v[ROWS][2];
#pragma unroll
        for (int u = 0; u < ROWS; ++u) load_row16(rows[u], lane, v[u]);
        float m = -INFINITY, l = 0.f, acc[16];
#pragma unroll
        for (int d = 0; d < 16; ++d) acc[d] = 0.f;
#pragma unroll
        for (int u = 0; u < ROWS; ++u) {
            const int i = warp + R128_WARPS * u;  // row within the group
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
            for (int w = 1; w < R128_WARPS; ++w) M = fmaxf(M, sm_m[w]);
            float L = 0.f, o0 = 0.f, o1 = 0.f;
            const int d0 = 2 * threadIdx.x;
#pragma unroll
            for (int w = 0; w < R128_WARPS; ++w) {
                const float f = expf(sm_m[w] - M);
                L = fmaf(f, sm_l[w], L);
                o0 = fmaf(f, sm_acc[w][d0], o0);
                o1 = fmaf(f, sm_acc[w][d0 + 1], o1);
            }
            const float inv = 1.f / L;
            uint8_t* dst = const_cast<uint8_t*>(row_addr(a.out, b, g, ROW_BYTES, a.status));
            if (dst) *reinterpret_cast<uint32_t*>(dst + d0 * 2) = pack_bf16x2(o0 * inv, o1 * inv);
        }
        __syncthreads();
    }
}

static DPaged to_dev(const HPaged& h) {
    DPaged d;
    d.base = static_cast<const uint8_t*>(h.base);
    d.pt = h.pt;
    d.pt_stride = h.pt_stride;
    d.page_stride = h.page_stride;
    d.n_pages = h.n_pages;
    d.rpp = h.rpp;
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
    a.status = h.status;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.stream = s;
    cfg.blockDim = dim3(h.ratio == 4 ? 256 : R128_WARPS * 32, 1, 1);
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
    if (h.ratio == 4) return cudaLaunchKernelEx(&cfg, compress_r4_kernel, a);
    return cudaLaunchKernelEx(&cfg, compress_r128_kernel, a);
}

}  // namespace csa
