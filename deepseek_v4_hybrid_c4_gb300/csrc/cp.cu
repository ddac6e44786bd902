// Context-parallel split of one long request's decode step ("SGLang 如何为 DeepSeek V4 打造
// 「Day-0」推理加速", sec. "3.1 长上下文预填充：Context Parallelism (CP)": each rank holds a share
// of the tokens, and the indexer's results meet in one exchange).  Each of R ranks scores a
// contiguous shard of the request's candidates and selects its local top k (csa_topk, sorted,
// with keys); after an all-gather of those R k-lists, every rank computes the exact global
// top k here; each rank then attends to the selected entries it holds (csa_sparse_attn_partial)
// and the partials meet in a log-sum-exp merge (csa_attn_merge).
//
// Why the merge is exact: an entry of the global top k is in its shard's top k (whatever
// ranks above it in its shard ranks above it globally), so the union of the local lists holds
// the global top k.  Ranks own increasing index ranges and each local list is sorted by
// (key desc, index asc), so in the rank-major concatenation equal keys appear in increasing
// global index order, and a select that breaks ties by position breaks them by global index.
#include "common.cuh"
#include "internal.h"

namespace csa {

// The fp32 score whose order-preserving key is `key` (the inverse of score_key; both zeros
// map to key 0x80000000, which comes back as +0).  Padding (key 0) comes back as a NaN with
// the sign set, whose key is 0 again: below every real score.
__device__ __forceinline__ float key_score(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

__global__ void __launch_bounds__(256) cp_keys_to_scores_kernel(const uint32_t* keys, int n, float* scores) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) scores[i] = key_score(keys[i]);
}

// Position p of the concatenation -> rank p / k, global index rank_lo[rank] + local index.
__global__ void __launch_bounds__(256) cp_map_kernel(TopkMergeLaunch a, const int32_t* pos, const uint32_t* pkeys) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= a.k) return;
    const int n = a.R * a.k;
    const int p = pos[i];
    if (p >= n) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    int64_t g = -1;
    if (p >= 0 && p < n) {
        const int r = p / a.k;
        const int32_t l = a.idx[p];
        const int64_t lo = __ldg(a.rank_lo + r), hi = __ldg(a.rank_lo + r + 1);
        if (l >= 0 && lo + l < hi) g = lo + l;
        else if (l >= 0) raise_status(a.status, CSA_ERR_DEVICE_BOUNDS);
    }
    if (a.idx_out) a.idx_out[i] = (int32_t)g;
    if (a.keys_out) a.keys_out[i] = g < 0 ? 0u : pkeys[i];
    if (a.sel_local) {
        const int64_t lo = __ldg(a.rank_lo + a.rank), hi = __ldg(a.rank_lo + a.rank + 1);
        a.sel_local[i] = (g >= lo && g < hi) ? (int32_t)(g - lo) : -1;
    }
}

struct TopkMergeLayout {
    size_t scores, hist, lists, pos, keys, total;
};
static TopkMergeLayout merge_layout(int R, int k) {
    const int64_t n = (int64_t)R * k;
    TopkMergeLayout L;
    size_t off = 0;
    L.scores = off;
    off += align_up((size_t)n * sizeof(float), 256);
    L.hist = off;
    off += align_up((size_t)kHistBlock * sizeof(uint32_t), 256);
    L.lists = off;
    off += align_up(select_set_lists_bytes(1, n), 256);
    L.pos = off;
    off += align_up((size_t)k * sizeof(int32_t), 256);
    L.keys = off;
    off += align_up((size_t)k * sizeof(uint32_t), 256);
    L.total = off;
    return L;
}

size_t topk_merge_workspace_bytes(int R, int k) { return merge_layout(R, k).total; }

cudaError_t launch_topk_merge(const TopkMergeLaunch& a, cudaStream_t s) {
    const int n = a.R * a.k;
    const TopkMergeLayout L = merge_layout(a.R, a.k);
    uint8_t* ws = static_cast<uint8_t*>(a.ws);
    float* scores = reinterpret_cast<float*>(ws + L.scores);
    int32_t* pos = reinterpret_cast<int32_t*>(ws + L.pos);
    uint32_t* pkeys = reinterpret_cast<uint32_t*>(ws + L.keys);
    cp_keys_to_scores_kernel<<<(n + 255) / 256, 256, 0, s>>>(a.keys, n, scores);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // the k best positions of the concatenation, by (score desc, position asc)
    SelectSetLaunch t;
    t.scores = scores;
    t.score_stride = 0;
    t.B = 1;
    t.max_G = n;
    t.n_tokens = nullptr;
    t.ratio = 1;
    t.k = a.k;
    t.idx_out = pos;
    t.hist = reinterpret_cast<uint32_t*>(ws + L.hist);
    t.lists = ws + L.lists;
    t.status = a.status;
    t.offsets = nullptr;
    t.G = n;
    t.standalone = true;
    t.keys_out = pkeys;
    e = launch_select_set(t, s, true);
    if (e != cudaSuccess) return e;
    cp_map_kernel<<<(a.k + 255) / 256, 256, 0, s>>>(a, pos, pkeys);
    return cudaGetLastError();
}

}  // namespace csa
