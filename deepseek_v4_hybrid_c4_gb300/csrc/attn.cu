// Stage 4: one attention over the selected compressed entries plus the sliding
// window of raw tokens, under a single softmax ("DeepSeek-V4 本地部署，SGLang 把活
// 做絕了", sec. "Kernel 層一堆狠活": SWA and the extra C4/C128 attention in one
// call; heads padded for the tensor-core tile as in "SGLang 如何为 DeepSeek V4
// 打造「Day-0」推理加速", sec. "3.2 高 TP 下的 FlashMLA 头填充").
//
//   l_j = scale * q_h . K_j,  o_h = sum_j softmax(l)_j V_j,  K = V = the bf16 latent row
//
// GB300 mapping.  One CTA = one 64-key tile range (a "split") x one half of the
// 512 V columns.  Heads are the MMA M dimension, padded to 128 (TMEM lane h =
// head h = thread h).  Per key tile:
//   gather 64 rows (cp.async 16 B, paged addressing) into a 128-byte-swizzled
//   K-major tile; S = Q K^T with tcgen05.mma (M=128, N=64, K=512) into TMEM;
//   each thread reads its head's 64 logits (tcgen05.ld), updates its running
//   max/sum (online softmax; the running max only moves when a tile raises it
//   by more than 2^8, then O is rescaled in TMEM); P (bf16) goes to shared memory;
//   O += P V with tcgen05.mma (M=128, N=256, K=64) where the same K tile is read
//   as an MN-major B operand.
// S uses TMEM columns [256, 320), the O half [0, 256).
//
// With one split per request the CTA writes the bf16 output directly.  Otherwise each
// split writes its rows normalised by their own sum (O_s / l_s as fp16: |values| <=
// max |V|, relative rounding 2^-11) and its (max, sum) to the workspace with coalesced
// stores (staged through shared memory), and a merge kernel (one CTA per head and
// request, chained by programmatic dependent launch) computes
// O = sum_s (l_s 2^(m_s - M) / L) (O_s / l_s) with every split's row loaded at once.
#include "common.cuh"
#include "internal.h"

namespace csa {

constexpr int AT_T = 128;                          // threads that own a TMEM lane (head row) each
constexpr int A1_T = 384;                          // attn_kernel: warps 4-11 only help gather and store
constexpr int AT_M = 128;
constexpr int AT_KT = 64;
constexpr int AT_DH = 256;
constexpr uint32_t SM_Q = 0;                       // 8 slabs x 128 rows x 128 B
constexpr uint32_t SM_K = 131072;                  // 8 slabs x 64 rows x 128 B
constexpr uint32_t SM_P = 196608;                  // 128 rows x 128 B
constexpr uint32_t SM_BAR = 212992;                // 2 mbarriers
constexpr uint32_t SM_TMEM = SM_BAR + 16;
constexpr uint32_t SM_KPTR = SM_BAR + 64;          // 64 row pointers
constexpr uint32_t SM_KOK = SM_KPTR + 64 * 8;      // 64-bit valid mask
constexpr uint32_t AT_SMEM = SM_KOK + 64 + 1024;   // + alignment slack
constexpr uint32_t R_PITCH = AT_DH * 2 + 16;       // staged fp16 row of one half (padded)
constexpr uint32_t SM_STG = 0;                     // this split's [128] staged rows (the Q tile's space)
constexpr int AT_MAX_SPLITS = 32;                  // splits per request (the merge holds them in registers)
constexpr uint32_t Q_SLAB = AT_M * 128;
constexpr uint32_t K_SLAB = AT_KT * 128;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;          // log2 units

struct AttnArgs {
    const uint16_t* q;
    int H;
    float sl2;                 // scale * log2(e)
    DPaged kc, kr;
    const int32_t* sel;
    int64_t sel_stride;
    int n_sel;
    const int64_t* n_tokens;
    int ratio;
    int nq;                    // decode: query positions per request
    const int64_t* n_done;     // decode, dense (sel == nullptr): compressed rows of earlier steps per
                               // request; rows [n_done, n_c) come from this step's compressor
    int64_t N;
    int swa;
    int tps, S;
    __half* part_o;            // [B][S][H][512] normalised partial rows (fp16)
    float2* part_ml;           // [B][2 halves][S][H] {max (log2 units), sum}
    uint16_t* out;
    float* lse;
    float* out_f32;            // mergeable partial: fp32 [B][H][512] normalised rows instead of out
    int32_t* status;
    DWorkSet kws;              // HiSparse working set of the compressed pool (table == nullptr: none)
};

// 2^x with the hardware's approximate exponential (ex2.approx.ftz: relative error below
// 2^-22, 2^-inf = +0); the softmax weights are graded by tolerance.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t chunk) {  // byte offset inside a 128-B-row slab
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

__global__ void __launch_bounds__(A1_T, 1) attn_kernel(AttnArgs a) {
    extern __shared__ uint8_t at_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int half = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
    const uint32_t bar_s = sbase + SM_BAR, bar_o = sbase + SM_BAR + 8;
    const uint8_t** kptr = reinterpret_cast<const uint8_t**>(sm + SM_KPTR);
    uint64_t* kok = reinterpret_cast<uint64_t*>(sm + SM_KOK);

    const int64_t N = a.n_tokens ? query_tokens(a.n_tokens, b, a.nq) : a.N;
    const int64_t W = N < a.swa ? N : a.swa;
    const int64_t n_c = a.sel ? a.n_sel : (a.n_tokens ? N / a.ratio : a.n_sel);
    const int64_t n_keys = n_c + W;
    const int64_t T = (n_keys + AT_KT - 1) / AT_KT;
    const int64_t t0 = (int64_t)split * a.tps;
    const int64_t t1 = t0 + a.tps < T ? t0 + a.tps : T;
    const int H = a.H;
    const int h = tid;  // head row owned by this thread

    const int S = a.S;
    float m_run = -INFINITY, l_run = 0.f;
    if (t0 >= t1) {
        pdl_wait();
        pdl_launch_dependents();
    }
    if (t0 < t1) {
        if (warp == 0) {
            tmem_alloc(sbase + SM_TMEM, 512);
            tmem_relinquish();
        }
        if (tid == 0) {
            mbar_init(bar_s, 1);
            mbar_init(bar_o, 1);
            fence_mbar_init();
        }
        // Q -> swizzled K-major tile (rows >= H are zero)
        const uint16_t* qb = a.q + (int64_t)b * H * D;
        for (int c = tid; c < AT_M * 64; c += A1_T) {
            const uint32_t row = c >> 6, ch = c & 63;
            const uint32_t dst = sbase + SM_Q + (ch >> 3) * Q_SLAB + swz(row, ch & 7);
            if ((int)row < H)
                cp_async16(dst, qb + row * D + ch * 8);
            else
                st_shared_zero16(dst);
        }
        // everything above touches only inputs of the step; the selection and the freshly
        // compressed rows come from the preceding kernels
        pdl_wait();
        pdl_launch_dependents();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + SM_TMEM);
        const uint32_t t_o = tmem;            // O half: columns [0, 256)
        const uint32_t t_s = tmem + AT_DH;    // S: columns [256, 320)
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        bool ok = true;

        // address of key j's row (selected compressed entry, then the window), or nullptr
        auto key_row = [&](int64_t j) -> const uint8_t* {
            if (j < n_c) {
                const int64_t g = a.sel ? (int64_t)__ldg(a.sel + (int64_t)b * a.sel_stride + j) : j;
                return g >= 0 ? ws_row(a.kws, a.kc, b, g, true, a.status) : nullptr;
            }
            if (j < n_keys) return row_addr(a.kr, b, N - W + (j - n_c), ROW_BYTES, a.status);
            return nullptr;
        };
        const uint8_t* p_next = tid < AT_KT ? key_row(t0 * AT_KT + tid) : nullptr;
        int it = 0;
        for (int64_t tile = t0; tile < t1; ++tile, ++it) {
            // ---- key rows of this tile (looked up while the previous tile was gathered)
            if (tid < AT_KT) {
                kptr[tid] = p_next;
                const unsigned m = __ballot_sync(0xffffffffu, p_next != nullptr);
                if (lane == 0) reinterpret_cast<uint32_t*>(kok)[warp] = m;
            }
            // the previous tile's P.V must be done before K/V and P are overwritten
            if (it > 0 && !mbar_wait(bar_o, (uint32_t)((it - 1) & 1))) ok = false;
            __syncthreads();
            // the rows slab-major, in four commit groups of two 128-byte slabs (the first group
            // also carries the staged Q), so that S runs on each pair of slabs as it lands
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                for (int c = tid; c < AT_KT * 16; c += A1_T) {
                    const uint32_t row = c >> 4, ch = 16 * g + (c & 15);
                    const uint32_t dst = sbase + SM_K + (ch >> 3) * K_SLAB + swz(row, ch & 7);
                    const uint8_t* src = kptr[row];
                    if (src)
                        cp_async16(dst, src + ch * 16);
                    else
                        st_shared_zero16(dst);
                }
                cp_async_commit();
            }
            // ---- S = Q K^T  (M=128, N=64, K=512: 8 slabs x 4 steps of 16), two slabs per group
            constexpr uint32_t id_s = idesc_bf16_f32(AT_M, AT_KT, false);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                if (g == 0) cp_async_wait_group<3>();
                else if (g == 1) cp_async_wait_group<2>();
                else if (g == 2) cp_async_wait_group<1>();
                else cp_async_wait_group<0>();
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int s = 2 * g; s < 2 * g + 2; ++s)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = sdesc_sw128(sbase + SM_Q + s * Q_SLAB + kk * 32, 16, 1024);
                            const uint64_t bd = sdesc_sw128(sbase + SM_K + s * K_SLAB + kk * 32, 16, 1024);
                            tc_mma_f16(t_s, ad, bd, id_s, (s | kk) ? 1u : 0u);
                        }
                    if (g == 3) tc_commit(bar_s);
                }
            }
            // the next tile's rows: look them up (dependent loads) while S runs
            if (tid < AT_KT && tile + 1 < t1) p_next = key_row((tile + 1) * AT_KT + tid);
            if (tid < AT_T) {  // ---- online softmax for row h (warps 0-3)
                if (!mbar_wait(bar_s, (uint32_t)(it & 1))) ok = false;
                tc_fence_after();
                uint32_t sr[2][32];
                tc_ld32(t_s + lane_off, sr[0]);
                tc_ld32(t_s + lane_off + 32, sr[1]);
                tc_wait_ld();
                const uint64_t valid = *kok;
                float x[64];
                float mt = -INFINITY;
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const bool v = (valid >> j) & 1ull;
                    x[j] = v ? __uint_as_float(sr[j >> 5][j & 31]) * a.sl2 : -INFINITY;
                    mt = fmaxf(mt, x[j]);
                }
                float alpha = 1.f;
                if (mt > -INFINITY) {
                    if (m_run == -INFINITY) {
                        m_run = mt;
                    } else if (mt > m_run + RESCALE_THRESHOLD) {
                        alpha = ex2(m_run - mt);
                        m_run = mt;
                    }
                }
                // rescale O (columns of this CTA's half) when the running max moved
                const bool need = it > 0 && alpha != 1.f;
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                    for (int c = 0; c < AT_DH; c += 32) {
                        uint32_t o[32];
                        tc_ld32(t_o + lane_off + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc_st32(t_o + lane_off + c, o);
                    }
                    tc_wait_st();
                }
                float lsum = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int j = 0; j < 64; j += 2) {
                    const float p0 = m_run == -INFINITY ? 0.f : ex2(x[j] - m_run);
                    const float p1 = m_run == -INFINITY ? 0.f : ex2(x[j + 1] - m_run);
                    const uint32_t w = pack_bf16x2(p0, p1);
                    pk[j >> 1] = w;
                    lsum += bf16lo(w) + bf16hi(w);
                }
                l_run = l_run * alpha + lsum;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_shared_v4(sbase + SM_P + swz((uint32_t)h, (uint32_t)c),
                                 make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncthreads();
            // ---- O += P V  (M=128, N=256, K=64: 4 steps of 16 keys); V read MN-major from the K tile
            if (tid == 0) {
                tc_fence_after();
                constexpr uint32_t id_o = idesc_bf16_f32(AT_M, AT_DH, true);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(sbase + SM_P + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(sbase + SM_K + (uint32_t)(half * 4) * K_SLAB + kk * 16 * 128,
                                                    K_SLAB, 1024);
                    tc_mma_f16(t_o, ad, bd, id_o, (it > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar_o);
            }
        }
        if (!mbar_wait(bar_o, (uint32_t)((it - 1) & 1))) ok = false;
        tc_fence_after();
        if (!ok && tid == 0) raise_status(a.status, CSA_ERR_TIMEOUT);
    }
    // ---- this split's rows, normalised (fp16 partial, or the bf16 output when S == 1), into
    //      shared memory (every MMA has completed, so the Q/K tiles' space is free), then
    //      coalesced to global memory
    const bool direct = S == 1 && !a.out_f32;
    if (t0 < t1) {
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + SM_TMEM);
        const uint32_t srow = sbase + SM_STG + (uint32_t)h * R_PITCH;
        for (int c0 = 0; c0 < AT_DH && tid < AT_T; c0 += 128) {  // four TMEM loads in flight, one wait
            uint32_t o[4][32];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
                tc_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(c0 + 32 * qq), o[qq]);
            tc_wait_ld();
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float f0 = __uint_as_float(o[qq][e + 2 * q]) * inv;
                        const float f1 = __uint_as_float(o[qq][e + 2 * q + 1]) * inv;
                        if (direct) {
                            w4[q] = pack_bf16x2(f0, f1);
                        } else {
                            const __half2 hv = __floats2half2_rn(f0, f1);
                            w4[q] = *reinterpret_cast<const uint32_t*>(&hv);
                        }
                    }
                    st_shared_v4(srow + (uint32_t)(c0 + 32 * qq + e) * 2u, make_uint4(w4[0], w4[1], w4[2], w4[3]));
                }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tmem, 512);
        // warp w copies rows w, w + 4, ...: one 512-byte row per warp instruction
        uint16_t* dst = direct ? a.out + (int64_t)b * H * D + half * AT_DH
                               : reinterpret_cast<uint16_t*>(a.part_o + ((int64_t)b * S + split) * H * D + half * AT_DH);
        constexpr int NWA = A1_T / 32;
        for (int r0 = warp; r0 < H; r0 += 8 * NWA) {  // eight rows per warp in flight
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = r0 + j * NWA;
                if (r < H) v[j] = ld_shared_v4(sbase + SM_STG + (uint32_t)r * R_PITCH + (uint32_t)lane * 16u);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int r = r0 + j * NWA;
                if (r < H) *reinterpret_cast<uint4*>(dst + (int64_t)r * D + lane * 8) = v[j];
            }
        }
    } else if (direct) {  // no keys at all
        for (int r = warp; r < H; r += A1_T / 32)
            *reinterpret_cast<uint4*>(a.out + ((int64_t)b * H + r) * D + half * AT_DH + lane * 8) = make_uint4(0, 0, 0, 0);
    }
    if (h < H) {
        const float l = t0 < t1 ? l_run : 0.f;
        if (!direct)
            a.part_ml[(((int64_t)b * 2 + half) * S + split) * H + h] = make_float2(m_run, l);
        else if (half == 0 && a.lse)
            a.lse[(int64_t)b * H + h] = l > 0.f ? (m_run + log2f(l)) * LN2 : -INFINITY;
    }
}

// ---------------------------------------------------------------- H <= 64
// With at most 64 heads, half of the M = 128 rows of every MMA would be padding.  One CTA
// then covers both V halves of a split, and the spare rows carry the second half:
//   O rows 0..63   += P V[:, 0:256]     O rows 64..127 += P V[:, 256:512]
// as one M=128, N=256, K=128 product [P 0; 0 P] [V_lo; V_hi]: eight K=16 steps, the first
// four with A = (P; 0) and B = the tile's first four slabs read MN-major, the last four with
// A = (0; P) and the other four slabs.  P sits between two zero blocks, so both A operands
// are windows of one 24 KiB region.  S = Q K^T keeps M = 128 with only Q's 64 rows staged
// (64 KiB): rows 64..127 of each slab's operand read the next slab, their logits land in
// TMEM lanes 64..127 and are never read.  The freed shared memory holds a second K tile:
// the next tile's rows are gathered while the current one is multiplied.
// TMEM: O [0, 256) (lane h: head h, columns 0..255; lane 64 + h: head h, columns 256..511),
// S [256, 320).
constexpr int A6_H = 64;
constexpr int A6_T = 384;  // warps 0-3 own the TMEM lane quarters (0-1 the softmax); warps 2-11 issue the row gathers
constexpr uint32_t A6_Q_SLAB = A6_H * 128;                  // 8 KiB
constexpr uint32_t A6_SM_Q = 0;                             // 8 slabs x 64 rows x 128 B
constexpr uint32_t A6_SM_K = 8 * A6_Q_SLAB;                 // 2 stages x 8 slabs x 64 rows x 128 B
constexpr uint32_t A6_KST = 8 * K_SLAB;                     // 64 KiB per stage
constexpr uint32_t A6_SM_P = A6_SM_K + 2 * A6_KST;          // [zero 8 KiB][P 8 KiB][zero 8 KiB]
constexpr uint32_t A6_SM_BAR = A6_SM_P + 3 * 8192;
constexpr uint32_t A6_SM_TMEM = A6_SM_BAR + 16;
constexpr uint32_t A6_SM_ALPHA = A6_SM_BAR + 64;            // [64] rescale factors, then [64] {m, l}
constexpr uint32_t A6_SM_ML = A6_SM_ALPHA + 64 * 4;
constexpr uint32_t A6_SM_KPTR = A6_SM_ML + 64 * 8;          // [2 stages][64] row pointers
constexpr uint32_t A6_SM_KOK = A6_SM_KPTR + 2 * 64 * 8;     // [2 stages] 64-bit valid masks
constexpr uint32_t A6_SMEM = A6_SM_KOK + 16 + 1024;         // + alignment slack
static_assert(A6_SMEM <= 227 * 1024, "attn64 shared memory");
static_assert(128 * R_PITCH <= A6_SM_P, "attn64 staging fits below P");

// A key's row address in two halves.  key_issue starts the page-table (and working-set) loads
// of a key whose selection entry is already in a register, without waiting for them;
// key_resolve turns them into the row's address, with the bounds check of row_addr.  Issued a
// tile ahead, the lookups of the tile after next run behind the current tile's products
// instead of stalling its softmax threads (behind the SM's row gathers, a lookup takes 1-2 us).
struct KeyRef {
    int64_t slot;  // row within its page
    int32_t pp;    // page id (the page table's entry; the logical page without a table)
    int32_t sl;    // working-set slot, or -1
    int32_t kind;  // 0: no key; 1: a compressed row (kc, kws); 2: a window row (kr)
};

__device__ __forceinline__ KeyRef key_issue(const AttnArgs& a, int b, int kind, int64_t r) {
    KeyRef k;
    k.kind = kind;
    k.sl = -1;
    k.pp = 0;
    k.slot = 0;
    if (kind == 0) return k;
    const DPaged& p = kind == 1 ? a.kc : a.kr;
    const int64_t lp = r / p.rpp;
    k.slot = r - lp * p.rpp;
    const int64_t e = (int64_t)(p.qpr > 1 ? b / p.qpr : b) * p.pt_stride + lp;
    if (kind == 1 && a.kws.table) {
        if (a.kws.touch) a.kws.touch[e] = a.kws.step;
        k.sl = a.kws.table[e];
    }
    k.pp = p.pt ? __ldg(p.pt + e) : (int32_t)lp;
    return k;
}

__device__ __forceinline__ const uint8_t* key_resolve(const AttnArgs& a, const KeyRef& k) {
    if (k.kind == 0) return nullptr;
    if (k.kind == 1 && a.kws.table && k.sl >= 0 && k.sl < a.kws.n_slots)
        return a.kws.base + k.sl * a.kc.page_stride + k.slot * (int64_t)ROW_BYTES;
    const DPaged& p = k.kind == 1 ? a.kc : a.kr;
    if (k.pp < 0 || k.pp >= p.n_pages) {
        raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
        return nullptr;
    }
    return p.base + k.pp * p.page_stride + k.slot * (int64_t)ROW_BYTES;
}

__global__ void __launch_bounds__(A6_T, 1) attn64_kernel(AttnArgs a) {
    extern __shared__ uint8_t at_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(at_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(sm);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, b = blockIdx.y;
    const uint32_t bar_s = sbase + A6_SM_BAR, bar_o = sbase + A6_SM_BAR + 8;
    const uint8_t** kptr = reinterpret_cast<const uint8_t**>(sm + A6_SM_KPTR);
    uint64_t* kok = reinterpret_cast<uint64_t*>(sm + A6_SM_KOK);
    float* sm_alpha = reinterpret_cast<float*>(sm + A6_SM_ALPHA);
    float2* sm_ml = reinterpret_cast<float2*>(sm + A6_SM_ML);

    const int64_t N = a.n_tokens ? query_tokens(a.n_tokens, b, a.nq) : a.N;
    const int64_t W = N < a.swa ? N : a.swa;
    const int64_t n_c = a.sel ? a.n_sel : (a.n_tokens ? N / a.ratio : a.n_sel);
    const int64_t n_keys = n_c + W;
    const int64_t T = (n_keys + AT_KT - 1) / AT_KT;
    const int64_t t0 = (int64_t)split * a.tps;
    const int64_t t1 = t0 + a.tps < T ? t0 + a.tps : T;
    const int H = a.H, S = a.S;
    const bool direct = S == 1 && !a.out_f32;
    const bool soft = tid < A6_H;  // warps 0, 1: head tid's softmax
    float m_run = -INFINITY, l_run = 0.f;

    if (t0 >= t1) {
        pdl_wait();
        pdl_launch_dependents();
        if (direct)  // no keys at all
            for (int r = warp; r < 2 * H; r += A6_T / 32)
                *reinterpret_cast<uint4*>(a.out + ((int64_t)b * H + (r >> 1)) * D + (r & 1) * AT_DH + lane * 8) =
                    make_uint4(0, 0, 0, 0);
        if (tid < H) {
            if (!direct) {
                const float2 z = make_float2(-INFINITY, 0.f);
                a.part_ml[(((int64_t)b * 2 + 0) * S + split) * H + tid] = z;
                a.part_ml[(((int64_t)b * 2 + 1) * S + split) * H + tid] = z;
            } else if (a.lse) {
                a.lse[(int64_t)b * H + tid] = -INFINITY;
            }
        }
        return;
    }
    if (warp == 0) {
        tmem_alloc(sbase + A6_SM_TMEM, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        fence_mbar_init();
    }
    // Q -> swizzled K-major tile of 64 rows (rows >= H are zero); the zero blocks around P
    const uint16_t* qb = a.q + (int64_t)b * H * D;
    for (int c = tid; c < A6_H * 64; c += A6_T) {
        const uint32_t row = c >> 6, ch = c & 63;
        const uint32_t dst = sbase + A6_SM_Q + (ch >> 3) * A6_Q_SLAB + swz(row, ch & 7);
        if ((int)row < H)
            cp_async16(dst, qb + row * D + ch * 8);
        else
            st_shared_zero16(dst);
    }
    for (int c = tid; c < 1024; c += A6_T)
        st_shared_zero16(sbase + A6_SM_P + (uint32_t)(c < 512 ? c : c + 512) * 16u);
    cp_async_commit();

    // key j: its selection entry (a load that nothing waits on until key_ref), then its lookups
    auto key_entry = [&](int64_t j) -> int64_t {
        return j < n_c && a.sel ? (int64_t)__ldg(a.sel + (int64_t)b * a.sel_stride + j) : j;
    };
    auto key_ref = [&](int64_t j, int64_t g) -> KeyRef {
        if (j < n_c) return key_issue(a, b, g >= 0 ? 1 : 0, g);
        return key_issue(a, b, j < n_keys ? 2 : 0, N - W + (j - n_c));
    };
    auto publish = [&](int st, const uint8_t* p) {  // warps 0, 1
        kptr[st * AT_KT + tid] = p;
        const unsigned m = __ballot_sync(0xffffffffu, p != nullptr);
        if (lane == 0) reinterpret_cast<uint32_t*>(kok + st)[warp] = m;
    };
    // Every thread but the softmax warps' (whose chain S -> softmax -> P V then runs while the
    // others are still held issuing copies into a full request queue); kptr[st] published and
    // visible.
    auto gather = [&](int st) {
        const uint32_t kb = sbase + A6_SM_K + (uint32_t)st * A6_KST;
        for (int c = tid - A6_H; c >= 0 && c < AT_KT * 64; c += A6_T - A6_H) {
            const uint32_t row = c >> 6, ch = c & 63;
            const uint32_t dst = kb + (ch >> 3) * K_SLAB + swz(row, ch & 7);
            const uint8_t* src = kptr[st * AT_KT + row];
            if (src)
                cp_async16(dst, src + ch * 16);
            else
                st_shared_zero16(dst);
        }
        cp_async_commit();
    };

    // The selection and the freshly compressed rows come from the preceding kernels.  A dense
    // step (no selection) needs them only from the first tile holding a row its compressor wrote,
    // so a split over earlier rows starts at once; everything else waits before its first tile.
    int64_t t_fresh = 0;  // the first tile that must wait for the preceding kernels
    if (!a.sel && a.n_tokens && a.n_done) {
        const int64_t done = __ldg(a.n_done + b / a.nq);
        t_fresh = done < n_c ? done / AT_KT : T;
    }
    bool waited = false;
    auto wait_for = [&](int64_t tile) {  // every thread, at the same points
        if (!waited && tile >= t_fresh) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
        }
    };
    if (t_fresh >= t1) pdl_launch_dependents();  // this split never waits (the merge waits for the grid)
    wait_for(t0);
    if (soft) {
        const int64_t j = t0 * AT_KT + tid;
        publish(0, key_resolve(a, key_ref(j, key_entry(j))));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    gather(0);
    // the lookups of the next tile, and the selection entries of the one after (a selection
    // is complete once the first wait returned; a dense split needs no entry loads)
    if (t0 + 1 < t1) wait_for(t0 + 1);
    KeyRef ref_next = {0, 0, -1, 0};
    if (soft && t0 + 1 < t1) {
        const int64_t j = (t0 + 1) * AT_KT + tid;
        ref_next = key_ref(j, key_entry(j));
    }
    int64_t g_after = soft && t0 + 2 < t1 ? key_entry((t0 + 2) * AT_KT + tid) : 0;
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(sm + A6_SM_TMEM);
    const uint32_t t_o = tmem, t_s = tmem + AT_DH;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    bool ok = true;
    int it = 0;
    for (int64_t tile = t0; tile < t1; ++tile, ++it) {
        const int st = it & 1;
        // P . V of the previous tile done: its K stage, P and O are free
        if (it > 0 && !mbar_wait(bar_o, (uint32_t)((it - 1) & 1))) ok = false;
        tc_fence_after();
        const bool more = tile + 1 < t1;
        if (soft && more) publish(st ^ 1, key_resolve(a, ref_next));
        cp_async_wait_all();  // this tile's rows (and Q) landed
        fence_proxy_async_smem();
        __syncthreads();
        // the lookups of the tile after next go out ahead of the next tile's rows
        if (soft && tile + 2 < t1) ref_next = key_ref((tile + 2) * AT_KT + tid, g_after);
        if (more) gather(st ^ 1);  // the next tile's rows, behind this tile's products
        // ---- S = Q K^T  (M=128, N=64, K=512); rows 64..127 are not used
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_s = idesc_bf16_f32(AT_M, AT_KT, false);
            const uint32_t kb = sbase + A6_SM_K + (uint32_t)st * A6_KST;
#pragma unroll
            for (int s8 = 0; s8 < 8; ++s8)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(sbase + A6_SM_Q + s8 * A6_Q_SLAB + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kb + s8 * K_SLAB + kk * 32, 16, 1024);
                    tc_mma_f16(t_s, ad, bd, id_s, (s8 | kk) ? 1u : 0u);
                }
            tc_commit(bar_s);
        }
        if (tile + 2 < t1) wait_for(tile + 2);  // before the gather of tile + 2 (fresh rows of a dense step)
        if (soft && tile + 3 < t1) g_after = key_entry((tile + 3) * AT_KT + tid);
        float alpha = 1.f;
        if (soft) {
            if (!mbar_wait(bar_s, (uint32_t)(it & 1))) ok = false;
            tc_fence_after();
            uint32_t sr[2][32];
            tc_ld32(t_s + lane_off, sr[0]);
            tc_ld32(t_s + lane_off + 32, sr[1]);
            tc_wait_ld();
            const uint64_t valid = kok[st];
            float x[64];
            float mt = -INFINITY;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                const bool v = (valid >> j) & 1ull;
                x[j] = v ? __uint_as_float(sr[j >> 5][j & 31]) * a.sl2 : -INFINITY;
                mt = fmaxf(mt, x[j]);
            }
            if (mt > -INFINITY) {
                if (m_run == -INFINITY) {
                    m_run = mt;
                } else if (mt > m_run + RESCALE_THRESHOLD) {
                    alpha = ex2(m_run - mt);
                    m_run = mt;
                }
            }
            float lsum = 0.f;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 64; j += 2) {
                const float p0 = m_run == -INFINITY ? 0.f : ex2(x[j] - m_run);
                const float p1 = m_run == -INFINITY ? 0.f : ex2(x[j + 1] - m_run);
                const uint32_t w = pack_bf16x2(p0, p1);
                pk[j >> 1] = w;
                lsum += bf16lo(w) + bf16hi(w);
            }
            l_run = l_run * alpha + lsum;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                st_shared_v4(sbase + A6_SM_P + 8192u + swz((uint32_t)tid, (uint32_t)c),
                             make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            sm_alpha[tid] = alpha;
        }
        __syncthreads();
        // rescale O (both column halves of the head) when its running max moved
        if (!soft && tid < AT_T) alpha = sm_alpha[tid - A6_H];
        if (tid < AT_T && it > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
            for (int c = 0; c < AT_DH; c += 32) {
                uint32_t o[32];
                tc_ld32(t_o + lane_off + c, o);
                tc_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                tc_st32(t_o + lane_off + c, o);
            }
            tc_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        // ---- O += [P 0; 0 P] [V_lo; V_hi]  (M=128, N=256, K=128)
        if (tid == 0) {
            tc_fence_after();
            constexpr uint32_t id_o = idesc_bf16_f32(AT_M, AT_DH, true);
            const uint32_t kb = sbase + A6_SM_K + (uint32_t)st * A6_KST;
#pragma unroll
            for (int hv = 0; hv < 2; ++hv)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = sdesc_sw128(sbase + A6_SM_P + (hv ? 0u : 8192u) + kk * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kb + (uint32_t)(hv * 4) * K_SLAB + kk * 16 * 128, K_SLAB, 1024);
                    tc_mma_f16(t_o, ad, bd, id_o, (it > 0 || hv > 0 || kk > 0) ? 1u : 0u);
                }
            tc_commit(bar_o);
        }
    }
    if (!mbar_wait(bar_o, (uint32_t)((it - 1) & 1))) ok = false;
    tc_fence_after();
    cp_async_wait_all();
    if (!ok && tid == 0) raise_status(a.status, CSA_ERR_TIMEOUT);
    if (soft) sm_ml[tid] = make_float2(m_run, l_run);
    __syncthreads();
    // ---- rows normalised (fp16 partial, or the bf16 output when S == 1), staged as
    //      row 2 * head + column half by warps 0-3, then coalesced to global memory by all
    if (tid < AT_T) {
        const int hd = tid & (A6_H - 1), hv = tid >> 6;
        const float l = sm_ml[hd].y;
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const uint32_t srow = sbase + (uint32_t)(2 * hd + hv) * R_PITCH;
        for (int c0 = 0; c0 < AT_DH; c0 += 128) {
            uint32_t o[4][32];
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) tc_ld32(t_o + lane_off + (uint32_t)(c0 + 32 * qq), o[qq]);
            tc_wait_ld();
#pragma unroll
            for (int qq = 0; qq < 4; ++qq)
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float f0 = __uint_as_float(o[qq][e + 2 * q]) * inv;
                        const float f1 = __uint_as_float(o[qq][e + 2 * q + 1]) * inv;
                        if (direct) {
                            w4[q] = pack_bf16x2(f0, f1);
                        } else {
                            const __half2 hh = __floats2half2_rn(f0, f1);
                            w4[q] = *reinterpret_cast<const uint32_t*>(&hh);
                        }
                    }
                    st_shared_v4(srow + (uint32_t)(c0 + 32 * qq + e) * 2u, make_uint4(w4[0], w4[1], w4[2], w4[3]));
                }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, 512);
    uint16_t* dst = direct ? a.out + (int64_t)b * H * D
                           : reinterpret_cast<uint16_t*>(a.part_o + ((int64_t)b * S + split) * H * D);
    constexpr int NWA = A6_T / 32;
    for (int r0 = warp; r0 < 2 * H; r0 += 8 * NWA) {  // eight 512-byte rows per warp in flight
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = r0 + j * NWA;
            if (r < 2 * H) v[j] = ld_shared_v4(sbase + (uint32_t)r * R_PITCH + (uint32_t)lane * 16u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = r0 + j * NWA;
            if (r < 2 * H) *reinterpret_cast<uint4*>(dst + (int64_t)(r >> 1) * D + (r & 1) * AT_DH + lane * 8) = v[j];
        }
    }
    if (tid < H) {
        if (!direct) {
            const float2 ml = make_float2(m_run, l_run);
            a.part_ml[(((int64_t)b * 2 + 0) * S + split) * H + tid] = ml;
            a.part_ml[(((int64_t)b * 2 + 1) * S + split) * H + tid] = ml;
        } else if (a.lse) {
            a.lse[(int64_t)b * H + tid] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
        }
    }
}

// Log-sum-exp merge of the splits: one CTA per (head, request); thread t owns columns
// 4t .. 4t+3 (half t / 64).  Every split's (max, sum) and row piece are loaded at once.
// Up to 16 splits every split's row piece and (max, sum) pair is loaded at once into registers
// (an instance for up to 8 splits holds half of them); above, the pairs go through shared
// memory, so that every row piece is still in flight at once within the registers that let
// four CTAs share an SM (a batch of 8 requests x 64 heads is 512 CTAs: one wave).
template <int MAXS>
__global__ void __launch_bounds__(128, MAXS > 16 ? 4 : 0) attn_merge_kernel(AttnArgs a) {
    pdl_wait();
    const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x;
    const int H = a.H, S = a.S, half = t >> 6;
    const float2* mlb = a.part_ml + ((int64_t)b * 2 + half) * S * H + h;
    const __half* pb = a.part_o + ((int64_t)b * S * H + h) * D + t * 4;
    float M = -INFINITY, L = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    float2 ml[MAXS];
    if constexpr (MAXS <= 16) {
        uint2 x[MAXS];
#pragma unroll
        for (int s = 0; s < MAXS; ++s) {
            if (s < S) {
                ml[s] = __ldcg(mlb + (int64_t)s * H);
                x[s] = __ldcg(reinterpret_cast<const uint2*>(pb + (int64_t)s * H * D));
            }
        }
#pragma unroll
        for (int s = 0; s < MAXS; ++s)
            if (s < S && ml[s].y > 0.f) M = fmaxf(M, ml[s].x);
#pragma unroll
        for (int s = 0; s < MAXS; ++s) {
            if (s < S && ml[s].y > 0.f) {
                const float w = ml[s].y * ex2(ml[s].x - M);
                const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&x[s].x));
                const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&x[s].y));
                L += w;
                o0 = fmaf(w, f01.x, o0);
                o1 = fmaf(w, f01.y, o1);
                o2 = fmaf(w, f23.x, o2);
                o3 = fmaf(w, f23.y, o3);
            }
        }
    } else {
        // the splits' (max, sum) pairs through shared memory (each half's 64 threads share them),
        // so that every split's row piece can be in flight at once in registers
        __shared__ float2 mls[2][MAXS];
        if ((t & 63) < S) mls[half][t & 63] = __ldcg(mlb + (int64_t)(t & 63) * H);
        uint2 x[MAXS];
#pragma unroll
        for (int s = 0; s < MAXS; ++s)
            if (s < S) x[s] = __ldcg(reinterpret_cast<const uint2*>(pb + (int64_t)s * H * D));
        __syncthreads();
#pragma unroll
        for (int s = 0; s < MAXS; ++s)
            if (s < S && mls[half][s].y > 0.f) M = fmaxf(M, mls[half][s].x);
#pragma unroll
        for (int s = 0; s < MAXS; ++s) {
            const float2 m2 = mls[half][s < S ? s : 0];
            if (s < S && m2.y > 0.f) {
                const float w = m2.y * ex2(m2.x - M);
                const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&x[s].x));
                const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&x[s].y));
                L += w;
                o0 = fmaf(w, f01.x, o0);
                o1 = fmaf(w, f01.y, o1);
                o2 = fmaf(w, f23.x, o2);
                o3 = fmaf(w, f23.y, o3);
            }
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    if (a.out_f32) {  // a mergeable partial: fp32 rows (zero when no key was attended)
        *reinterpret_cast<float4*>(a.out_f32 + ((int64_t)b * H + h) * D + t * 4) =
            make_float4(o0 * inv, o1 * inv, o2 * inv, o3 * inv);
    } else {
        uint2 r;
        r.x = pack_bf16x2(o0 * inv, o1 * inv);
        r.y = pack_bf16x2(o2 * inv, o3 * inv);
        *reinterpret_cast<uint2*>(a.out + ((int64_t)b * H + h) * D + t * 4) = r;
    }
    if (t == 0 && a.lse) a.lse[(int64_t)b * H + h] = L > 0.f ? (M + log2f(L)) * LN2 : -INFINITY;
}

// Log-sum-exp merge of R partial attentions of the same heads over disjoint key sets (each a
// normalised fp32 row O_r and its natural-log lse_r; lse_r = -inf for an empty set):
//   L = sum_r e^(lse_r - M), O = sum_r e^(lse_r - M) O_r / L, lse = M + ln L,  M = max_r lse_r.
// One CTA per head, thread t owns columns 4t .. 4t+3; the partials are read in rank order.
__global__ void __launch_bounds__(128) attn_lse_merge_kernel(const float* o_parts, const float* lse_parts, int R, int H,
                                                             uint16_t* out, float* lse) {
    const int h = blockIdx.x, t = threadIdx.x;
    float M = -INFINITY;
    for (int r = 0; r < R; ++r) M = fmaxf(M, __ldg(lse_parts + (int64_t)r * H + h));
    float L = 0.f, o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    if (M > -INFINITY) {
        for (int r = 0; r < R; ++r) {
            const float lr = __ldg(lse_parts + (int64_t)r * H + h);
            if (!(lr > -INFINITY)) continue;
            const float w = expf(lr - M);
            const float4 v = __ldg(reinterpret_cast<const float4*>(o_parts + ((int64_t)r * H + h) * D) + t);
            L += w;
            o0 = fmaf(w, v.x, o0);
            o1 = fmaf(w, v.y, o1);
            o2 = fmaf(w, v.z, o2);
            o3 = fmaf(w, v.w, o3);
        }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint2 rr;
    rr.x = pack_bf16x2(o0 * inv, o1 * inv);
    rr.y = pack_bf16x2(o2 * inv, o3 * inv);
    *reinterpret_cast<uint2*>(out + (int64_t)h * D + t * 4) = rr;
    if (t == 0 && lse) lse[h] = L > 0.f ? M + logf(L) : -INFINITY;
}

cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int R, int H, void* out, float* lse,
                             cudaStream_t s) {
    attn_lse_merge_kernel<<<H, 128, 0, s>>>(o_parts, lse_parts, R, H, static_cast<uint16_t*>(out), lse);
    return cudaGetLastError();
}

// Split heuristic (device independent so workspace sizes are stable): about one wave
// of CTAs (one per SM) on 152 SMs -- 2*B*S of them above 64 heads (one per V half), B*S
// at or below -- with at most one split per key tile.
static void plan_splits(int B, int H, int64_t max_keys, int* tps, int* S) {
    const int64_t T = (max_keys + AT_KT - 1) / AT_KT;
    const bool h64 = H <= A6_H;
    int64_t s = (h64 ? 152 : 76) / (B > 0 ? B : 1);
    if (s < 1) s = 1;
    if (s > (h64 ? AT_MAX_SPLITS : 16)) s = h64 ? AT_MAX_SPLITS : 16;
    if (s > T) s = T;
    if (s < 1) s = 1;
    int64_t t = (T + s - 1) / s;
    if (t < 1) t = 1;
    s = (T + t - 1) / t;
    if (s < 1) s = 1;
    *tps = (int)t;
    *S = (int)s;
}

size_t attn_workspace_bytes(int B, int H, int64_t max_keys) {
    int tps, S;
    plan_splits(B, H, max_keys, &tps, &S);
    const size_t po = (size_t)B * S * H * D * sizeof(__half);
    const size_t pm = (size_t)B * 2 * S * H * sizeof(float2);
    return ((po + 255) & ~size_t(255)) + pm;
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

cudaError_t launch_attn(const AttnLaunch& h, cudaStream_t s, bool pdl) {
    AttnArgs a;
    a.q = static_cast<const uint16_t*>(h.q);
    a.H = h.H;
    a.sl2 = h.scale * LOG2E;
    a.kc = to_dev(h.kv_c);
    a.kr = to_dev(h.kv_raw);
    a.sel = h.sel;
    a.sel_stride = h.sel_stride;
    a.n_sel = h.n_sel;
    a.n_tokens = h.n_tokens;
    a.ratio = h.ratio;
    a.nq = h.nq > 1 ? h.nq : 1;
    a.n_done = h.n_done;
    a.N = h.N;
    a.swa = h.swa;
    plan_splits(h.B, h.H, h.max_keys, &a.tps, &a.S);
    const size_t po = (size_t)h.B * a.S * h.H * D * sizeof(__half);
    a.part_o = static_cast<__half*>(h.ws);
    a.part_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(h.ws) + ((po + 255) & ~size_t(255)));
    a.out = static_cast<uint16_t*>(h.out);
    a.out_f32 = h.out_f32;
    a.lse = h.lse;
    a.status = h.status;
    a.kws.table = h.hs.table;
    a.kws.base = static_cast<uint8_t*>(h.hs.base);
    a.kws.n_slots = h.hs.n_slots;
    a.kws.touch = h.hs.touch;
    a.kws.step = h.hs.step;
    {
        cudaError_t e = set_func_attr_once((const void*)attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)AT_SMEM);
        if (e == cudaSuccess)
            e = set_func_attr_once((const void*)attn64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)A6_SMEM);
        if (e != cudaSuccess) return e;
    }
    const bool h64 = h.H <= A6_H;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cfg.gridDim = h64 ? dim3((unsigned)a.S, (unsigned)h.B, 1) : dim3(2, (unsigned)a.S, (unsigned)h.B);
    cfg.blockDim = dim3(h64 ? A6_T : A1_T, 1, 1);
    cfg.dynamicSmemBytes = h64 ? A6_SMEM : AT_SMEM;
    cfg.stream = s;
    cudaError_t e = h64 ? cudaLaunchKernelEx(&cfg, attn64_kernel, a) : cudaLaunchKernelEx(&cfg, attn_kernel, a);
    if (e != cudaSuccess || (a.S == 1 && !a.out_f32)) return e;
    cfg.numAttrs = 1;  // the merge waits for the attention grid (griddepcontrol.wait)
    cfg.gridDim = dim3((unsigned)h.H, (unsigned)h.B, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    // up to 8 splits: 48 registers, so that eleven CTAs share an SM (the 32-request batch of 64
    // heads, 2,048 CTAs of 5 splits, in little more than one wave instead of three); up to 10
    // (a 1M request's 640 keys): 56 registers, eight CTAs per SM, so that the 384-512 merge CTAs
    // of a speculative verify fit beside the attention's CTAs
    return a.S <= 8    ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<8>, a)
           : a.S <= 10 ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<10>, a)
           : a.S <= 16 ? cudaLaunchKernelEx(&cfg, attn_merge_kernel<16>, a)
                       : cudaLaunchKernelEx(&cfg, attn_merge_kernel<AT_MAX_SPLITS>, a);
}

}  // namespace csa
