// Host-side launchers shared between the libcsa translation units.
#pragma once
#include <cuda_runtime.h>
#include <cstdint>

#include "csa.h"

namespace csa {

constexpr int kLatentRowBytes = 1024;  // one bf16 latent row (512 dims)
constexpr int kHistBins = 2048;        // first top-k digit: key >> 21
// Per-request top-k block in the workspace, cleared before every step: one histogram per radix
// digit (six of kHistBins counters; digit 0 first), or, after the tensor-core bounds, one
// histogram of up to 2^14 bins.
constexpr int kHistBlock = 8 * kHistBins;
// Bits of the lower bounds' first digit after the tensor-core bounds, by query positions per
// request (the score kernel keeps n_q such histograms in shared memory).
inline int bound_hist_bits(int nq) { return nq <= 1 ? 14 : (nq == 2 ? 13 : 12); }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Per-device launch facts, safe to call from several host threads and on several devices:
// the current device's SM count (0 on failure), and a kernel attribute set per device
// (cudaFuncSetAttribute applies to the current device only) -- again whenever the value asked for
// differs from the one it holds, a call with the value it holds costing nothing.
int device_sm_count();
cudaError_t set_func_attr_once(const void* func, cudaFuncAttribute attr, int value);

struct HWorkSet {          // HiSparse working set of a pool (see DWorkSet); table == nullptr: none
    const int32_t* table = nullptr;
    void* base = nullptr;
    int64_t n_slots = 0;
    uint32_t* touch = nullptr;
    uint32_t step = 0;
};

struct HPaged {            // host copy of a paged buffer description (see csa_paged)
    const void* base;
    const int32_t* pt;     // device page table(s) or nullptr
    int64_t pt_stride;     // entries between requests' tables
    int64_t page_stride;   // bytes
    int64_t n_pages;
    int32_t rpp;
    int32_t qpr = 1;       // batch entries per page table (speculative verify: query positions)
};

// Stage 1.  Single mode (n_tokens == nullptr): groups [first, first + count) of one
// sequence.  Batched mode: request b = blockIdx.y compresses [n_done[b], n_tokens[b]/ratio).
// hist_zero (nullable): [B][kHistBlock] blocks whose first hist_words words block (0, b) clears
// for stages 2 and 3 (the histograms the chosen select uses).
struct CompressLaunch {
    HWorkSet hs;               // HiSparse: the compressed pool's GPU working set (optional)
    int nq = 1;                // decode: query positions per request (speculative verify)
    HPaged raw, out;
    const float* w_gate;
    const float* b_pos;
    int ratio;
    int B;
    const int64_t* n_tokens;
    const int64_t* n_done;
    int64_t first, count;
    uint32_t* hist_zero;
    int hist_words = kHistBlock;
    int carveout = cudaSharedmemCarveoutDefault;  // C4 decode: the shared-memory carveout asked for
    int32_t* status;
    const void* ring_pool = nullptr;  // batched mode: pending tokens from per-request rings
    const int32_t* ring_page = nullptr;
    int32_t ring_size = 0;
    int64_t ring_n_pages = 0;
};
cudaError_t launch_compress(const CompressLaunch& a, cudaStream_t s, bool pdl);

// Stage 2.  Single mode (n_tokens == nullptr): one sequence of G candidates.
// Batched: request b has n_tokens[b] / ratio candidates; scores at b * score_stride.
struct ScoreLaunch {
    int nq = 1;                // decode: query positions per request (speculative verify)
    const void* q_idx;     // bf16 [B, Hi, 128]
    const float* w_h;      // fp32 [B, Hi]
    int Hi;
    HPaged kidx;
    bool fp8;
    float* scores;
    int64_t score_stride;
    int B;
    const int64_t* n_tokens;
    int ratio;
    int64_t G;             // single mode
    int64_t max_G;         // host bound (grid sizing)
    uint32_t* hist;        // fused first-digit histogram, [B][kHistBlock] (zeroed beforehand), or nullptr
    int32_t* status;
    int reserve = 0;       // CTA slots left free for a kernel running beside this one (the decode
                           // compressor's warp holds one SM's second slot while the score kernel starts)
};
cudaError_t launch_score(const ScoreLaunch& a, cudaStream_t s, bool pdl);
// The TMA tensor map (a CUtensorMap at `map`) of an index-key pool seen as [pages][rows per
// page][128 dims], box 16 rows x 128 B, 128-byte swizzle; false when it cannot be encoded.
bool make_kidx_map(void* map, const HPaged& p, bool fp8, int64_t rows_per_page, int64_t n_pages);
// Stage 2 on the tensor cores, bf16 keys: for every candidate a bracket [lower, upper] that holds
// the fixed-order score (upper to `scores`, lower to `lower` when set), and, with hist, the first
// digit of the lower bounds' keys.  Needs Hi <= 16, nq <= 4.
bool score_bound_supported(int Hi, int nq, bool fp8);
// Words of each batch entry's histogram block that a decode step's select uses: the six digit
// histograms of the wide select, or the 2^bound_hist_bits(nq) bins after the bounds.
constexpr int kWideSelectHistWords = 6 * kHistBins;
cudaError_t launch_score_bound(const ScoreLaunch& a, float* lower, cudaStream_t s, bool pdl);

// Stage 3.  Request b's scores: single: [0, G); offsets mode: [offsets[b], offsets[b+1]);
// decode mode: b * score_stride + [0, n_tokens[b] / ratio).  hist: [B][kHistBlock], zeroed
// before the launch; with hist_fused its first kHistBins words hold digit 0's histogram
// from stage 2, otherwise the select counts digit 0 itself.
struct TopkLaunch {
    int nq = 1;                // decode: query positions per request (speculative verify)
    const float* scores;
    int B;
    int64_t G;                 // single mode
    int64_t max_G;             // host bound on every request's length (grid sizing)
    const int64_t* offsets;    // offsets mode
    const int64_t* n_tokens;   // decode mode
    int ratio;
    int64_t score_stride;
    int k;
    int32_t* idx_out;          // [B, k]
    uint32_t* keys_out;        // [B, k] or nullptr
    bool sorted;               // true: by (score desc, index asc); false: the set in a fixed order
    bool hist_fused;
    uint32_t* hist;
    int32_t* status;
};
size_t topk_lists_bytes(int B, int64_t max_G, int k);
cudaError_t launch_topk(const TopkLaunch& a, cudaStream_t s, bool pdl);

// Stage 3 in the decode step: the top-k set of request b's scores b * score_stride +
// [0, n_tokens[b] / ratio), with the first digit's histogram from stage 2 in hist ([B]
// [kHistBlock], zeroed before stage 2).  lists: select_set_lists_bytes(B, max_G) bytes of
// workspace.  Only where select_set_supported(max_G, k).
struct SelectSetLaunch {
    int nq = 1;                // decode: query positions per request (speculative verify)
    const float* scores;
    int64_t score_stride;      // a multiple of 4
    int B;
    int64_t max_G;
    const int64_t* n_tokens;   // decode mode; else offsets mode (offsets) or single (G)
    int ratio;
    int k;
    int32_t* idx_out;          // [B, k]
    uint32_t* hist;
    void* lists;
    int32_t* status;
    const int64_t* offsets = nullptr;
    int64_t G = 0;
    // standalone: the first digit's histogram is counted here (hist zeroed beforehand) and
    // the set is sorted by (score desc, index asc) at the end, keys to keys_out when given
    bool standalone = false;
    uint32_t* keys_out = nullptr;
};
bool select_set_supported(int64_t max_G, int k);
// Stage 3 after launch_score_bound: scores hold the upper bounds and hist the lower bounds'
// first digit; the candidates the bounds cannot rule out are rescored in the fixed order from
// the query and the bf16 key rows, then an exact top-k picks the set (ascending index order).
// Decode mode only.
struct BoundRescore {
    const void* q_idx;         // bf16 [B, Hi, 128]
    const float* w_h;          // fp32 [B, Hi]
    int Hi;
    HPaged kidx;               // bf16 rows of 256 B
};
cudaError_t launch_select_bound(const SelectSetLaunch& a, const BoundRescore& r, cudaStream_t s, bool pdl);
size_t select_set_lists_bytes(int B, int64_t max_G);
cudaError_t launch_select_set(const SelectSetLaunch& a, cudaStream_t s, bool pdl);

// Stage 4 (+ log-sum-exp merge).  Per request b: keys = sel rows of kv_c (n_sel of
// them, -1 = padding; sel == nullptr: rows 0..n_c-1 with n_c = n_tokens/ratio in
// decode mode or n_sel in single mode) followed by the last min(swa, N) raw rows.
struct AttnLaunch {
    HWorkSet hs;               // HiSparse: the compressed pool's GPU working set (optional)
    int nq = 1;                // decode: query positions per request (speculative verify)
    const void* q;             // bf16 [B, H, 512]
    int H;
    float scale;
    HPaged kv_c, kv_raw;
    const int32_t* sel;        // [B, sel_stride] or nullptr (dense)
    int64_t sel_stride;
    int n_sel;                 // sparse: selection length; dense single: number of rows
    int B;
    const int64_t* n_tokens;   // decode mode (device) or nullptr
    int ratio;
    int64_t N;                 // single mode: raw tokens
    int64_t max_keys;          // host bound on keys per request
    int swa;
    void* out;                 // bf16 [B, H, 512]
    float* lse;                // [B, H] or nullptr
    float* out_f32 = nullptr;  // instead of out: fp32 [B, H, 512] rows of a mergeable partial
    const int64_t* n_done = nullptr;  // decode, dense: rows of earlier steps per request (see attn.cu)
    void* ws;
    size_t ws_bytes;
    int32_t* status;
};
size_t attn_workspace_bytes(int B, int H, int64_t max_keys);
// this device's sticky status word (the kernels' status argument)
int32_t* device_status_ptr();
cudaError_t launch_attn(const AttnLaunch& a, cudaStream_t s, bool pdl);
// Log-sum-exp merge of R partials (fp32 rows [R][H][512], natural-log lse [R][H]) into bf16
// out [H][512] and lse [H] (nullable).
cudaError_t launch_lse_merge(const float* o_parts, const float* lse_parts, int R, int H, void* out, float* lse,
                             cudaStream_t s);
// Context-parallel global top-k: the k best of R ranks' sorted local top-k lists (keys, indices
// local to each rank's range), as global indices and as rows of one rank's range.
struct TopkMergeLaunch {
    const uint32_t* keys;      // [R * k]
    const int32_t* idx;        // [R * k] indices local to rank p / k's range, < 0: padding
    const int64_t* rank_lo;    // device [R + 1]: rank r holds global candidates [rank_lo[r], rank_lo[r+1])
    int R, k;
    int rank;                  // the rank whose rows sel_local lists (-1: none)
    int32_t* sel_local;        // [k] or nullptr
    int32_t* idx_out;          // [k] or nullptr
    uint32_t* keys_out;        // [k] or nullptr
    void* ws;
    int32_t* status;
};
size_t topk_merge_workspace_bytes(int R, int k);
cudaError_t launch_topk_merge(const TopkMergeLaunch& a, cudaStream_t s);

}  // namespace csa
