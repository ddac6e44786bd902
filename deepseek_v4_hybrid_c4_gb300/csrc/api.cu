// libcsa C ABI: argument validation, workspace layout and the launch sequence of
// each entry point (see include/csa.h for the contract of every call).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "csa.h"
#include "internal.h"

namespace csa {

// Sticky per-device status word: kernels OR error bits into it.
__device__ int32_t g_status_word;

constexpr int kMaxDevices = 64;
static int32_t* g_status_ptr[kMaxDevices];
static std::mutex g_status_mu;

static int32_t* status_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_status_mu);
    if (!g_status_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        g_status_ptr[dev] = static_cast<int32_t*>(p);
    }
    return g_status_ptr[dev];
}

int32_t* device_status_ptr() { return status_ptr(); }

struct AttrDone {
    const void* func;
    cudaFuncAttribute attr;
    int value;
};
static std::vector<AttrDone> g_attr_done[kMaxDevices];
static int g_sm_count[kMaxDevices];
static std::mutex g_launch_mu;

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_launch_mu);
    if (!g_sm_count[dev] &&
        cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        g_sm_count[dev] = 0;
    return g_sm_count[dev];
}

cudaError_t set_func_attr_once(const void* func, cudaFuncAttribute attr, int value) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_launch_mu);
    AttrDone* cur = nullptr;  // the value this attribute holds now, if set here before
    for (AttrDone& d : g_attr_done[dev])
        if (d.func == func && d.attr == attr) cur = &d;
    if (cur && cur->value == value) return cudaSuccess;
    e = cudaFuncSetAttribute(func, attr, value);
    if (e != cudaSuccess) return e;
    if (cur) cur->value = value;
    else g_attr_done[dev].push_back({func, attr, value});
    return cudaSuccess;
}


// Query positions per request from which the decode step scores through the tensor-core bounds.
constexpr int kBoundMinQueries = 2;

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool al4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

static csa_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? CSA_OK : CSA_ERR_CUDA;
}

static csa_status check_paged(const csa_paged& p, int row_bytes) {
    if (!p.base || !al16(p.base)) return CSA_ERR_INVALID_ARG;
    if (p.rows_per_page < 1 || p.page_stride_bytes % 16 || p.n_pages < 1) return CSA_ERR_INVALID_ARG;
    if ((int64_t)p.rows_per_page * row_bytes > p.page_stride_bytes) return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

static HPaged host_paged(const csa_paged& p) {
    HPaged h;
    h.base = p.base;
    h.pt = p.page_table;
    h.pt_stride = 0;
    h.page_stride = p.page_stride_bytes;
    h.n_pages = p.n_pages;
    h.rpp = p.rows_per_page;
    return h;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace csa

using namespace csa;

extern "C" {

int32_t csa_version(void) { return 100; }

const char* csa_status_string(csa_status s) {
    switch (s) {
        case CSA_OK: return "ok";
        case CSA_ERR_INVALID_ARG: return "invalid argument";
        case CSA_ERR_UNSUPPORTED: return "unsupported shape or parameter";
        case CSA_ERR_CUDA: return "CUDA error";
        case CSA_ERR_TIMEOUT: return "device wait timed out";
        case CSA_ERR_DEVICE_BOUNDS: return "device bounds check failed";
        case CSA_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

csa_status csa_read_device_status(void* stream, int32_t* out) {
    if (!out) return CSA_ERR_INVALID_ARG;
    int32_t* p = status_ptr();
    if (!p) return CSA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(int32_t), s) != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return CSA_ERR_CUDA;
    *out = v;
    return CSA_OK;
}

csa_status csa_compress(csa_paged kv_raw, int64_t n_tokens, int32_t ratio, const float* w_gate, const float* b_pos,
                        int64_t first_group, int64_t n_groups, csa_paged kv_c_out, void* stream) {
    if (ratio != 4 && ratio != 128) return CSA_ERR_UNSUPPORTED;
    if (check_paged(kv_raw, kLatentRowBytes) || check_paged(kv_c_out, kLatentRowBytes)) return CSA_ERR_INVALID_ARG;
    if (!w_gate || !b_pos || !al16(w_gate) || !al4(b_pos)) return CSA_ERR_INVALID_ARG;
    if (n_tokens < 0 || first_group < 0 || n_groups < 0 || (first_group + n_groups) * ratio > n_tokens)
        return CSA_ERR_INVALID_ARG;
    if (n_groups == 0) return CSA_OK;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    CompressLaunch c;
    c.raw = host_paged(kv_raw);
    c.out = host_paged(kv_c_out);
    c.w_gate = w_gate;
    c.b_pos = b_pos;
    c.ratio = ratio;
    c.B = 1;
    c.n_tokens = nullptr;
    c.n_done = nullptr;
    c.first = first_group;
    c.count = n_groups;
    c.hist_zero = nullptr;
    c.status = st;
    return from_cuda(launch_compress(c, static_cast<cudaStream_t>(stream), false));
}

csa_status csa_index_score(const void* q_idx, const float* w_h, int32_t Hi, csa_paged k_idx, csa_dtype k_dtype,
                           int64_t G, float* scores, void* stream) {
    if (Hi < 1 || Hi > 16) return CSA_ERR_UNSUPPORTED;
    if (k_dtype != CSA_BF16 && k_dtype != CSA_FP8_E4M3) return CSA_ERR_UNSUPPORTED;
    const int rb = k_dtype == CSA_BF16 ? 256 : 128;
    if (!q_idx || !al16(q_idx) || !w_h || !al4(w_h) || !scores || !al4(scores)) return CSA_ERR_INVALID_ARG;
    if (check_paged(k_idx, rb)) return CSA_ERR_INVALID_ARG;
    if (G < 0 || G > 0x7FFFFFFFLL) return CSA_ERR_INVALID_ARG;
    if (k_idx.page_table && k_idx.rows_per_page % 16) return CSA_ERR_UNSUPPORTED;
    if (G == 0) return CSA_OK;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    ScoreLaunch l;
    l.q_idx = q_idx;
    l.w_h = w_h;
    l.Hi = Hi;
    l.kidx = host_paged(k_idx);
    if (!k_idx.page_table) {  // contiguous rows: one logical page holds everything
        l.kidx.rpp = 1 << 30;
        l.kidx.page_stride = 0;
        l.kidx.n_pages = 1;
    }
    l.fp8 = k_dtype == CSA_FP8_E4M3;
    l.scores = scores;
    l.score_stride = 0;
    l.B = 1;
    l.n_tokens = nullptr;
    l.ratio = 4;
    l.G = G;
    l.max_G = G;
    l.hist = nullptr;
    l.status = st;
    return from_cuda(launch_score(l, static_cast<cudaStream_t>(stream), false));
}

csa_status csa_index_score_bounds(const void* q_idx, const float* w_h, int32_t Hi, csa_paged k_idx, csa_dtype k_dtype,
                                  int64_t G, float* lower, float* upper, void* stream) {
    if (Hi < 1 || Hi > 16) return CSA_ERR_UNSUPPORTED;
    if (k_dtype != CSA_BF16) return CSA_ERR_UNSUPPORTED;
    if (!q_idx || !al16(q_idx) || !w_h || !al4(w_h) || !upper || !al4(upper) || (lower && !al4(lower)))
        return CSA_ERR_INVALID_ARG;
    if (check_paged(k_idx, 256)) return CSA_ERR_INVALID_ARG;
    if (G < 0 || G > 0x7FFFFFFFLL) return CSA_ERR_INVALID_ARG;
    if (k_idx.page_table && k_idx.rows_per_page % 16) return CSA_ERR_UNSUPPORTED;
    if (G == 0) return CSA_OK;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    ScoreLaunch l;
    l.q_idx = q_idx;
    l.w_h = w_h;
    l.Hi = Hi;
    l.kidx = host_paged(k_idx);
    if (!k_idx.page_table) {  // contiguous rows: one logical page holds everything
        l.kidx.rpp = 1 << 30;
        l.kidx.page_stride = 0;
        l.kidx.n_pages = 1;
    }
    l.fp8 = false;
    l.scores = upper;
    l.score_stride = 0;
    l.B = 1;
    l.n_tokens = nullptr;
    l.ratio = 4;
    l.G = G;
    l.max_G = G;
    l.hist = nullptr;
    l.status = st;
    return from_cuda(launch_score_bound(l, lower, static_cast<cudaStream_t>(stream), false));
}

size_t csa_topk_workspace_size(int32_t B, int64_t max_G, int32_t k) {
    if (B < 1 || B > 65535 || max_G < 0 || max_G > 0x7FFFFFFFLL || k < 1 || k > 2048) return 0;
    // one histogram per radix digit, then (wide select) every scan CTA's lists and counts
    return align256((size_t)B * kHistBlock * sizeof(uint32_t)) +
           (select_set_supported(max_G, k) ? select_set_lists_bytes(B, max_G) : 0);
}

static csa_status topk_common(const float* scores, const int64_t* offsets, int32_t B, int64_t G, int32_t k,
                              int32_t* idx_out, uint32_t* keys_out, void* workspace, size_t ws_bytes,
                              void* stream) {
    if (k < 1 || k > 2048) return CSA_ERR_UNSUPPORTED;
    if (!scores || !al4(scores) || !idx_out || !al4(idx_out)) return CSA_ERR_INVALID_ARG;
    if (keys_out && !al4(keys_out)) return CSA_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || G < 0 || G > 0x7FFFFFFFLL) return CSA_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < csa_topk_workspace_size(B, G, k) || !al16(workspace)) return CSA_ERR_WORKSPACE;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    TopkLaunch t;
    t.scores = scores;
    t.B = B;
    t.G = G;
    t.max_G = G;
    t.offsets = offsets;
    t.n_tokens = nullptr;
    t.ratio = 1;
    t.score_stride = 0;
    t.k = k;
    t.idx_out = idx_out;
    t.keys_out = keys_out;
    t.sorted = true;
    t.hist_fused = false;
    t.hist = static_cast<uint32_t*>(workspace);
    t.status = st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (select_set_supported(G, k)) {  // wide select: clear, first digit, scan, sorted finish (no memset)
        SelectSetLaunch w;
        w.scores = scores;
        w.score_stride = 0;
        w.B = B;
        w.max_G = G;
        w.n_tokens = nullptr;
        w.ratio = 1;
        w.k = k;
        w.idx_out = idx_out;
        w.hist = static_cast<uint32_t*>(workspace);
        w.lists = static_cast<uint8_t*>(workspace) + align256((size_t)B * kHistBlock * sizeof(uint32_t));
        w.status = st;
        w.offsets = offsets;
        w.G = G;
        w.standalone = true;
        w.keys_out = keys_out;
        e = launch_select_set(w, s, true);
    } else {  // one cluster per request; its histograms live in the cluster's shared memory
        e = launch_topk(t, s, false);
    }
    return from_cuda(e);
}

csa_status csa_topk(const float* scores, int64_t G, int32_t k, int32_t* idx_out, uint32_t* keys_out,
                    void* workspace, size_t ws_bytes, void* stream) {
    return topk_common(scores, nullptr, 1, G, k, idx_out, keys_out, workspace, ws_bytes, stream);
}

csa_status csa_topk_batched(const float* scores, const int64_t* offsets, int32_t B, int64_t max_G, int32_t k,
                            int32_t* idx_out, uint32_t* keys_out, void* workspace, size_t ws_bytes,
                            void* stream) {
    if (!offsets) return CSA_ERR_INVALID_ARG;
    return topk_common(scores, offsets, B, max_G, k, idx_out, keys_out, workspace, ws_bytes, stream);
}

csa_status csa_topk_cluster(const float* scores, const int64_t* offsets, int32_t B, int64_t max_G, int32_t k,
                            int32_t* idx_out, uint32_t* keys_out, void* stream) {
    if (k < 1 || k > 2048) return CSA_ERR_UNSUPPORTED;
    if (!scores || !al4(scores) || !idx_out || !al4(idx_out)) return CSA_ERR_INVALID_ARG;
    if (keys_out && !al4(keys_out)) return CSA_ERR_INVALID_ARG;
    if (B < 1 || B > 65535 || max_G < 0 || max_G > 0x7FFFFFFFLL) return CSA_ERR_INVALID_ARG;
    if (!offsets && B != 1) return CSA_ERR_INVALID_ARG;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    TopkLaunch t;
    t.scores = scores;
    t.B = B;
    t.G = max_G;
    t.max_G = max_G;
    t.offsets = offsets;
    t.n_tokens = nullptr;
    t.ratio = 1;
    t.score_stride = 0;
    t.k = k;
    t.idx_out = idx_out;
    t.keys_out = keys_out;
    t.sorted = true;
    t.hist_fused = false;
    t.hist = nullptr;
    t.status = st;
    return from_cuda(launch_topk(t, static_cast<cudaStream_t>(stream), false));
}

size_t csa_sparse_attn_workspace_size(int32_t H, int32_t n_sel, int32_t swa) {
    if (H < 1 || n_sel < 0 || swa < 0) return 0;
    return attn_workspace_bytes(1, H, (int64_t)n_sel + swa);
}

csa_status csa_sparse_attn(const void* q, int32_t H, float scale, csa_paged kv_c, const int32_t* sel, int32_t n_sel,
                           csa_paged kv_raw, int64_t n_tokens, int32_t swa, void* out, float* lse, void* workspace,
                           size_t ws_bytes, void* stream) {
    if (H < 1 || H > 128 || swa < 0 || swa > 128) return CSA_ERR_UNSUPPORTED;
    if (!q || !al16(q) || !out || !al16(out) || (lse && !al4(lse)) || (sel && !al4(sel))) return CSA_ERR_INVALID_ARG;
    if (n_sel < 0 || n_tokens < 0) return CSA_ERR_INVALID_ARG;
    const int64_t W = n_tokens < swa ? n_tokens : swa;
    if (n_sel + W < 1) return CSA_ERR_INVALID_ARG;
    if (n_sel > 0 && check_paged(kv_c, kLatentRowBytes)) return CSA_ERR_INVALID_ARG;
    if (W > 0 && check_paged(kv_raw, kLatentRowBytes)) return CSA_ERR_INVALID_ARG;
    const size_t need = attn_workspace_bytes(1, H, n_sel + W);
    if (need > 0 && (!workspace || ws_bytes < need || !al16(workspace))) return CSA_ERR_WORKSPACE;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    AttnLaunch a;
    a.q = q;
    a.H = H;
    a.scale = scale;
    a.kv_c = host_paged(kv_c);
    a.kv_raw = host_paged(kv_raw);
    a.sel = sel;
    a.sel_stride = 0;
    a.n_sel = n_sel;
    a.B = 1;
    a.n_tokens = nullptr;
    a.ratio = 4;
    a.N = n_tokens;
    a.max_keys = n_sel + W;
    a.swa = swa;
    a.out = out;
    a.lse = lse;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.status = st;
    return from_cuda(launch_attn(a, static_cast<cudaStream_t>(stream), false));
}

// ------------------------------------------------------------------ context-parallel pieces
csa_status csa_sparse_attn_partial(const void* q, int32_t H, float scale, csa_paged kv_c, const int32_t* sel,
                                   int32_t n_sel, csa_paged kv_raw, int64_t n_tokens, int32_t swa, float* o_part,
                                   float* lse_part, void* workspace, size_t ws_bytes, void* stream) {
    if (H < 1 || H > 128 || swa < 0 || swa > 128) return CSA_ERR_UNSUPPORTED;
    if (!q || !al16(q) || !o_part || !al16(o_part) || !lse_part || !al4(lse_part) || (sel && !al4(sel)))
        return CSA_ERR_INVALID_ARG;
    if (n_sel < 0 || n_tokens < 0 || (n_sel > 0 && !sel)) return CSA_ERR_INVALID_ARG;
    const int64_t W = n_tokens < swa ? n_tokens : swa;
    if (n_sel > 0 && check_paged(kv_c, kLatentRowBytes)) return CSA_ERR_INVALID_ARG;
    if (W > 0 && check_paged(kv_raw, kLatentRowBytes)) return CSA_ERR_INVALID_ARG;
    const size_t need = attn_workspace_bytes(1, H, n_sel + W);
    if (!workspace || ws_bytes < need || !al16(workspace)) return CSA_ERR_WORKSPACE;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    AttnLaunch a;
    a.q = q;
    a.H = H;
    a.scale = scale;
    a.kv_c = host_paged(kv_c);
    a.kv_raw = host_paged(kv_raw);
    a.sel = sel;
    a.sel_stride = 0;
    a.n_sel = n_sel;
    a.B = 1;
    a.n_tokens = nullptr;
    a.ratio = 4;
    a.N = n_tokens;
    a.max_keys = n_sel + W;
    a.swa = swa;
    a.out = nullptr;
    a.out_f32 = o_part;
    a.lse = lse_part;
    a.ws = workspace;
    a.ws_bytes = ws_bytes;
    a.status = st;
    return from_cuda(launch_attn(a, static_cast<cudaStream_t>(stream), false));
}

csa_status csa_attn_merge(const float* o_parts, const float* lse_parts, int32_t R, int32_t H, void* out, float* lse,
                          void* stream) {
    if (H < 1 || H > 128 || R < 1) return CSA_ERR_UNSUPPORTED;
    if (!o_parts || !al16(o_parts) || !lse_parts || !al4(lse_parts) || !out || !al16(out) || (lse && !al4(lse)))
        return CSA_ERR_INVALID_ARG;
    return from_cuda(launch_lse_merge(o_parts, lse_parts, R, H, out, lse, static_cast<cudaStream_t>(stream)));
}

size_t csa_topk_merge_workspace_size(int32_t R, int32_t k) {
    if (R < 1 || k < 1 || k > 2048 || (int64_t)R * k > 4194304) return 0;
    return topk_merge_workspace_bytes(R, k);
}

csa_status csa_topk_merge(const uint32_t* keys, const int32_t* idx, const int64_t* rank_lo, int32_t R, int32_t k,
                          int32_t rank, int32_t* sel_local, int32_t* idx_out, uint32_t* keys_out, void* workspace,
                          size_t ws_bytes, void* stream) {
    if (k < 1 || k > 2048 || R < 1 || (int64_t)R * k > 4194304) return CSA_ERR_UNSUPPORTED;
    if (!keys || !al4(keys) || !idx || !al4(idx) || !rank_lo || (reinterpret_cast<uintptr_t>(rank_lo) & 7u))
        return CSA_ERR_INVALID_ARG;
    if ((sel_local && !al4(sel_local)) || (idx_out && !al4(idx_out)) || (keys_out && !al4(keys_out)))
        return CSA_ERR_INVALID_ARG;
    if (sel_local && (rank < 0 || rank >= R)) return CSA_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < topk_merge_workspace_bytes(R, k) || !al16(workspace)) return CSA_ERR_WORKSPACE;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    TopkMergeLaunch m;
    m.keys = keys;
    m.idx = idx;
    m.rank_lo = rank_lo;
    m.R = R;
    m.k = k;
    m.rank = sel_local ? rank : -1;
    m.sel_local = sel_local;
    m.idx_out = idx_out;
    m.keys_out = keys_out;
    m.ws = workspace;
    m.status = st;
    return from_cuda(launch_topk_merge(m, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ fused decode
struct DecodeLayout {
    size_t scores, hist, lists, sel, attn, total;
    int64_t score_stride;
};

static int decode_nq(const csa_decode_params* p) { return p->n_q > 1 ? p->n_q : 1; }

static csa_status decode_check(const csa_decode_params* p) {
    if (!p) return CSA_ERR_INVALID_ARG;
    if (p->n_q < 0 || p->n_q > 16 || (int64_t)p->B * decode_nq(p) > 65535) return CSA_ERR_UNSUPPORTED;
    if (p->ratio != 4 && p->ratio != 128) return CSA_ERR_UNSUPPORTED;
    if (p->B < 1 || p->B > 65535 || p->H < 1 || p->H > 128 || p->swa < 0 || p->swa > 128)
        return CSA_ERR_UNSUPPORTED;
    if (p->max_tokens < p->ratio) return CSA_ERR_INVALID_ARG;
    if (!p->n_tokens || !p->n_groups_done || !p->kv_raw || !p->kv_c || !p->page_table || !p->w_gate || !p->b_pos ||
        !p->q || !p->out)
        return CSA_ERR_INVALID_ARG;
    if (!al16(p->kv_raw) || !al16(p->kv_c) || !al16(p->q) || !al16(p->out) || !al16(p->w_gate))
        return CSA_ERR_INVALID_ARG;
    if (p->raw_rows_per_page < 1 || p->raw_page_stride % 16 || p->c_page_stride % 16 || p->n_pages < 1)
        return CSA_ERR_INVALID_ARG;
    if ((int64_t)p->raw_rows_per_page * 1024 > p->raw_page_stride) return CSA_ERR_INVALID_ARG;
    const int c_rpp = p->c_page_table ? p->c_rows_per_page : p->raw_rows_per_page / p->ratio;
    if (!p->c_page_table && p->raw_rows_per_page % p->ratio) return CSA_ERR_UNSUPPORTED;
    if (c_rpp < 1 || (int64_t)c_rpp * 1024 > p->c_page_stride) return CSA_ERR_INVALID_ARG;
    if (p->c_page_table && p->c_n_pages < 1) return CSA_ERR_INVALID_ARG;
    if (p->hs_ws_pool) {  // HiSparse: C4 only, explicit compressed paging
        if (p->ratio != 4) return CSA_ERR_UNSUPPORTED;
        if (!p->c_page_table || !p->hs_ws_table || p->hs_n_slots < 1 || p->hs_n_slots > 0x7FFFFFFF ||
            !al16(p->hs_ws_pool))
            return CSA_ERR_INVALID_ARG;
    }
    if (p->ring_pool) {
        if (!al16(p->ring_pool) || !p->ring_page || p->ring_n_pages < 1) return CSA_ERR_INVALID_ARG;
        if (p->ring_size < p->ratio || p->ring_size % p->ratio) return CSA_ERR_INVALID_ARG;
    }
    if (p->ratio == 4) {
        if (p->Hi < 1 || p->Hi > 16 || p->k < 1 || p->k > 2048) return CSA_ERR_UNSUPPORTED;
        if (p->k_dtype != CSA_BF16 && p->k_dtype != CSA_FP8_E4M3) return CSA_ERR_UNSUPPORTED;
        if (!p->k_idx || !p->q_idx || !p->w_h || !al16(p->k_idx) || !al16(p->q_idx)) return CSA_ERR_INVALID_ARG;
        const int rb = p->k_dtype == CSA_BF16 ? 256 : 128;
        if (p->kidx_page_stride % 16 || (int64_t)c_rpp * rb > p->kidx_page_stride) return CSA_ERR_INVALID_ARG;
        if (c_rpp % 16) return CSA_ERR_UNSUPPORTED;
    }
    return CSA_OK;
}

static DecodeLayout decode_layout(const csa_decode_params* p) {
    DecodeLayout L;
    const int64_t max_G = p->max_tokens / p->ratio;
    const int Bq = p->B * decode_nq(p);  // batch entries: (request, query position)
    L.score_stride = (max_G + 3) & ~int64_t(3);
    size_t off = 0;
    L.scores = off;
    if (p->ratio == 4) off += align256((size_t)Bq * L.score_stride * sizeof(float));
    L.hist = off;
    if (p->ratio == 4) off += align256((size_t)Bq * kHistBlock * sizeof(uint32_t));
    L.lists = off;
    if (p->ratio == 4)
        off += align256(select_set_supported(max_G, p->k) ? select_set_lists_bytes(Bq, max_G)
                                                          : topk_lists_bytes(Bq, max_G, p->k));
    L.sel = off;
    if (p->ratio == 4 && !p->sel) off += align256((size_t)Bq * p->k * sizeof(int32_t));
    L.attn = off;
    const int64_t W = p->max_tokens < p->swa ? p->max_tokens : p->swa;
    const int64_t max_keys = (p->ratio == 4 ? p->k : max_G) + W;
    off += align256(attn_workspace_bytes(Bq, p->H, max_keys));
    L.total = off > 256 ? off : 256;  // never 0: a size of 0 means the parameters were rejected
    return L;
}

size_t csa_decode_workspace_size(const csa_decode_params* p) {
    if (decode_check(p) != CSA_OK) return 0;
    return decode_layout(p).total;
}

csa_status csa_decode(const csa_decode_params* p, void* workspace, size_t ws_bytes, void* stream) {
    return csa_decode_timed(p, workspace, ws_bytes, stream, nullptr);
}

csa_status csa_decode_timed(const csa_decode_params* p, void* workspace, size_t ws_bytes, void* stream,
                            void* const* ev) {
    csa_status rc = decode_check(p);
    if (rc) return rc;
    const DecodeLayout L = decode_layout(p);
    if (L.total > 0 && (!workspace || ws_bytes < L.total || !al16(workspace))) return CSA_ERR_WORKSPACE;
    int32_t* st = status_ptr();
    if (!st) return CSA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const int64_t max_G = p->max_tokens / p->ratio;
    const int nq = decode_nq(p);
    const int Bq = p->B * nq;  // stages 2-4 run per (request, query position)
    auto mark = [&](int i) {
        if (ev && ev[i]) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
    };
    mark(0);

    HPaged raw;
    raw.base = p->kv_raw;
    raw.pt = p->page_table;
    raw.pt_stride = p->page_table_stride;
    raw.page_stride = p->raw_page_stride;
    raw.n_pages = p->n_pages;
    raw.rpp = p->raw_rows_per_page;
    HPaged cp;
    cp.base = p->kv_c;
    cp.pt = p->c_page_table ? p->c_page_table : p->page_table;
    cp.pt_stride = p->c_page_table ? p->c_page_table_stride : p->page_table_stride;
    cp.page_stride = p->c_page_stride;
    cp.n_pages = p->c_page_table ? p->c_n_pages : p->n_pages;
    cp.rpp = p->c_page_table ? p->c_rows_per_page : p->raw_rows_per_page / p->ratio;
    uint32_t* hist = p->ratio == 4 ? reinterpret_cast<uint32_t*>(ws + L.hist) : nullptr;
    // Speculative verify with bf16 keys: one pass over the keys for every query position,
    // brackets on the tensor cores, exact rescoring of the candidates they leave open.  (With one
    // position the fixed-order kernel and the shorter select win: 1M step 40.6 against 52.5 us;
    // from two positions the pass does: 48.4 against 63.9 us back to back.)
    const bool bound = p->ratio == 4 && nq >= kBoundMinQueries && p->k_dtype == CSA_BF16 &&
                       score_bound_supported(p->Hi, nq, false) && select_set_supported(max_G, p->k);

    // 1. compress the completed groups that are not in the pool yet (and clear the histogram)
    CompressLaunch c;
    c.raw = raw;
    c.out = cp;
    c.w_gate = p->w_gate;
    c.b_pos = p->b_pos;
    c.ratio = p->ratio;
    c.B = p->B;
    c.n_tokens = p->n_tokens;
    c.n_done = p->n_groups_done;
    c.first = 0;
    c.count = 0;
    c.hist_zero = hist;
    c.hist_words = bound ? 1 << bound_hist_bits(nq) : kWideSelectHistWords;
    // bf16 keys: the score kernel's CTAs fill the SM's shared memory (two of about 100 KB, or one
    // of about 200 KB), so the compressor's SM takes the largest carveout too
    c.carveout = p->k_dtype == CSA_BF16 ? (int)cudaSharedmemCarveoutMaxShared : (int)cudaSharedmemCarveoutDefault;
    c.status = st;
    c.ring_pool = p->ring_pool;
    c.ring_page = p->ring_page;
    c.ring_size = p->ring_size;
    c.ring_n_pages = p->ring_n_pages;
    c.nq = nq;
    if (p->hs_ws_pool) {  // new rows go to the mirror and, when resident, to the working set
        c.hs.table = p->hs_ws_table;
        c.hs.base = p->hs_ws_pool;
        c.hs.n_slots = p->hs_n_slots;
    }
    cudaError_t e = launch_compress(c, s, false);
    if (e != cudaSuccess) return CSA_ERR_CUDA;
    mark(1);

    const int32_t* sel = nullptr;
    if (p->ratio == 4) {
        // 2. index scores of every candidate (+ the first radix digit's histogram)
        ScoreLaunch l;
        l.q_idx = p->q_idx;
        l.w_h = p->w_h;
        l.Hi = p->Hi;
        l.kidx = cp;
        l.kidx.base = p->k_idx;
        l.kidx.page_stride = p->kidx_page_stride;
        l.fp8 = p->k_dtype == CSA_FP8_E4M3;
        l.scores = reinterpret_cast<float*>(ws + L.scores);
        l.score_stride = L.score_stride;
        l.B = Bq;
        l.nq = nq;
        l.kidx.qpr = nq;
        l.n_tokens = p->n_tokens;
        l.ratio = p->ratio;
        l.G = 0;
        l.max_G = max_G;
        l.hist = hist;
        l.status = st;
        l.reserve = Bq == 1 ? 1 : 0;  // the compressor's single warp, which starts just ahead
        e = bound ? launch_score_bound(l, nullptr, s, ev == nullptr) : launch_score(l, s, ev == nullptr);
        if (e != cudaSuccess) return CSA_ERR_CUDA;
        mark(2);
        // 3. top-k per request
        int32_t* sel_out = p->sel ? p->sel : reinterpret_cast<int32_t*>(ws + L.sel);
        if (bound) {
            SelectSetLaunch t;
            t.scores = l.scores;
            t.score_stride = L.score_stride;
            t.B = Bq;
            t.nq = nq;
            t.max_G = max_G;
            t.n_tokens = p->n_tokens;
            t.ratio = p->ratio;
            t.k = p->k;
            t.idx_out = sel_out;
            t.hist = hist;
            t.lists = ws + L.lists;
            t.status = st;
            BoundRescore r;
            r.q_idx = p->q_idx;
            r.w_h = p->w_h;
            r.Hi = p->Hi;
            r.kidx = l.kidx;
            e = launch_select_bound(t, r, s, ev == nullptr);
        } else if (select_set_supported(max_G, p->k)) {
            SelectSetLaunch t;
            t.scores = l.scores;
            t.score_stride = L.score_stride;
            t.B = Bq;
            t.nq = nq;
            t.max_G = max_G;
            t.n_tokens = p->n_tokens;
            t.ratio = p->ratio;
            t.k = p->k;
            t.idx_out = sel_out;
            t.hist = hist;
            t.lists = ws + L.lists;
            t.status = st;
            e = launch_select_set(t, s, ev == nullptr);
        } else {
            TopkLaunch t;
            t.scores = l.scores;
            t.B = Bq;
            t.nq = nq;
            t.G = 0;
            t.max_G = max_G;
            t.offsets = nullptr;
            t.n_tokens = p->n_tokens;
            t.ratio = p->ratio;
            t.score_stride = L.score_stride;
            t.k = p->k;
            t.idx_out = sel_out;
            t.keys_out = nullptr;
            t.sorted = false;  // attention takes the set; a fixed order keeps the step deterministic
            t.hist_fused = true;
            t.hist = hist;
            t.status = st;
            e = launch_topk(t, s, ev == nullptr);
        }
        if (e != cudaSuccess) return CSA_ERR_CUDA;
        mark(3);
        sel = sel_out;
    } else {
        mark(2);
        mark(3);
    }
    // 4. attention over selection (or every compressed entry) + SWA
    AttnLaunch a;
    a.q = p->q;
    a.H = p->H;
    a.scale = p->scale;
    a.kv_c = cp;
    a.kv_raw = raw;
    a.kv_c.qpr = nq;
    a.kv_raw.qpr = nq;
    a.nq = nq;
    if (p->hs_ws_pool) {  // resident pages from the working set, the others from the mirror
        a.hs.table = p->hs_ws_table;
        a.hs.base = p->hs_ws_pool;
        a.hs.n_slots = p->hs_n_slots;
        a.hs.touch = p->hs_touch;
        a.hs.step = p->hs_step;
    }
    a.sel = sel;
    a.n_done = p->n_groups_done;
    a.sel_stride = p->k;
    a.n_sel = p->ratio == 4 ? p->k : 0;
    a.B = Bq;
    a.n_tokens = p->n_tokens;
    a.ratio = p->ratio;
    a.N = 0;
    const int64_t W = p->max_tokens < p->swa ? p->max_tokens : p->swa;
    a.max_keys = (p->ratio == 4 ? p->k : max_G) + W;
    a.swa = p->swa;
    a.out = p->out;
    a.lse = p->lse;
    a.ws = ws + L.attn;
    a.ws_bytes = L.total - L.attn;
    a.status = st;
    e = launch_attn(a, s, ev == nullptr);
    mark(4);
    return from_cuda(e);
}

}  // extern "C"
