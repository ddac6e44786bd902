// HiSparse coordinator: the GPU working set of the C4 compressed pool, whose full copy lives in
// host memory ("DeepSeek-V4 本地部署，SGLang 把活做絕了", sec. "HiSparse：把不活躍 KV 甩到 CPU":
// a CPU-pinned mirror of the C4 pool, a small GPU working set, pages swapped every step by a
// coordinator with LRU eviction; "SGLang 如何为 DeepSeek V4 打造「Day-0」推理加速", sec.
// "创新 3：HiSparse": GPU miss -> swap-in from the CPU mirror).
//
// GB300 mapping.  The decode step never waits for a swap: a page that is not resident is read
// by the attention straight from the mirror (pinned host memory, read through NVLink-C2C), and
// the step stamps every page it read.  Between steps the coordinator reads the stamps back,
// decides on the host which pages to bring in (LRU over the slots), and one gather kernel copies
// those pages from the mirror into their slots; the new residency table follows on the stream.
// The asynchronous form (collect, then apply one or more steps later) keeps the host and the
// swap off the decode stream: the evictions are published on it, the copies and the installs
// run on a side stream beside the next steps.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "internal.h"

struct csa_hisparse {
    int32_t B = 0;
    int64_t stride = 0;             // logical pages per request (the compressed page table's stride)
    int64_t n_slots = 0;
    std::vector<int32_t> table;     // [B * stride]: slot or -1
    std::vector<int64_t> owner;     // [n_slots]: table entry held, or -1
    std::vector<uint32_t> stamp;    // [n_slots]: the last step that read the slot's page
    std::vector<uint32_t> touch;    // host copy of the step's stamps
    std::vector<int32_t> plan;      // host copy of the last plan (request, logical page, slot)
    int32_t* d_plan = nullptr;      // device copy, n_slots triples
    // asynchronous form (csa_hisparse_collect / csa_hisparse_apply): pinned host buffers and events
    uint32_t* h_touch = nullptr;    // [B * stride] stamps read back by collect
    uint32_t collected_step = 0;    // the step those stamps belong to
    bool collected = false;
    int32_t* h_table_evict = nullptr;    // [B * stride] the table with this plan's evictions only
    int32_t* h_table_install = nullptr;  // [B * stride] the table with the plan's pages installed
    int32_t* h_plan = nullptr;           // [3 * n_slots] the plan, for its upload
    cudaEvent_t ev_touch = nullptr;      // the stamps have landed in h_touch
    cudaEvent_t ev_evict = nullptr;      // the evictions are in the device table (decode stream)
    cudaEvent_t ev_swap = nullptr;       // the last apply's swap and installs are done (side stream)
    bool swap_pending = false;
};

namespace csa {

// One CTA per planned page: page_stride bytes from the mirror page of (request, logical page)
// into the slot, 16 bytes per thread and load.
__global__ void __launch_bounds__(256) hisparse_swap_kernel(const int32_t* plan, const uint8_t* mirror,
                                                            const int32_t* pt, int64_t pt_stride, int64_t n_pages,
                                                            int64_t page_stride, uint8_t* slots, int32_t* status) {
    const int32_t b = plan[3 * blockIdx.x], lp = plan[3 * blockIdx.x + 1], sl = plan[3 * blockIdx.x + 2];
    const int64_t page = __ldg(pt + (int64_t)b * pt_stride + lp);
    if (page < 0 || page >= n_pages) {
        if (threadIdx.x == 0) raise_status(status, CSA_ERR_DEVICE_BOUNDS);
        return;
    }
    const uint4* src = reinterpret_cast<const uint4*>(mirror + page * page_stride);
    uint4* dst = reinterpret_cast<uint4*>(slots + (int64_t)sl * page_stride);
    for (int64_t i = threadIdx.x; i < page_stride / 16; i += blockDim.x) dst[i] = src[i];
}

}  // namespace csa

using namespace csa;

extern "C" {

csa_status csa_hisparse_create(int32_t B, int64_t table_stride, int64_t n_slots, csa_hisparse** out) {
    if (!out) return CSA_ERR_INVALID_ARG;
    *out = nullptr;
    if (B < 1 || table_stride < 1 || n_slots < 1 || n_slots > 0x7FFFFFFF) return CSA_ERR_INVALID_ARG;
    csa_hisparse* h = new (std::nothrow) csa_hisparse;
    if (!h) return CSA_ERR_CUDA;
    h->B = B;
    h->stride = table_stride;
    h->n_slots = n_slots;
    h->table.assign((size_t)B * table_stride, -1);
    h->owner.assign((size_t)n_slots, -1);
    h->stamp.assign((size_t)n_slots, 0u);
    h->touch.assign((size_t)B * table_stride, 0u);
    *out = h;  // the device plan buffer comes with the first update (planning alone needs no GPU)
    return CSA_OK;
}

void csa_hisparse_destroy(csa_hisparse* h) {
    if (!h) return;
    if (h->swap_pending) cudaEventSynchronize(h->ev_swap);
    cudaFree(h->d_plan);
    cudaFreeHost(h->h_touch);
    cudaFreeHost(h->h_table_evict);
    cudaFreeHost(h->h_table_install);
    cudaFreeHost(h->h_plan);
    if (h->ev_touch) cudaEventDestroy(h->ev_touch);
    if (h->ev_evict) cudaEventDestroy(h->ev_evict);
    if (h->ev_swap) cudaEventDestroy(h->ev_swap);
    delete h;
}

const int32_t* csa_hisparse_table(const csa_hisparse* h) { return h ? h->table.data() : nullptr; }

// The LRU plan (see csa_hisparse_plan).  With grow_from (nullable), page lp of request b is
// never brought in when lp >= grow_from[b]: a page that can still receive compressed rows.
static csa_status plan_impl(csa_hisparse* h, const uint32_t* touch, uint32_t step, int32_t* plan, int64_t max_plan,
                            int64_t* n_in, int64_t* n_evicted, const int64_t* grow_from) {
    const int64_t n = (int64_t)h->B * h->stride;
    // the step's resident pages are refreshed first, so that none of them is evicted below
    bool missed = false;
    for (int64_t e = 0; e < n; ++e) {
        if (touch[e] != step) continue;
        if (h->table[e] >= 0)
            h->stamp[h->table[e]] = step;
        else if (!grow_from || e % h->stride < grow_from[e / h->stride])
            missed = true;
    }
    if (!missed || max_plan == 0) {  // every page the step read is resident (or may not come in)
        if (n_in) *n_in = 0;
        if (n_evicted) *n_evicted = 0;
        return CSA_OK;
    }
    // candidates: free slots in order, then resident slots by (stamp, slot), never this step's
    std::vector<int64_t> cand;
    cand.reserve((size_t)h->n_slots);
    for (int64_t s = 0; s < h->n_slots; ++s)
        if (h->owner[s] < 0) cand.push_back(s);
    const size_t n_free = cand.size();
    for (int64_t s = 0; s < h->n_slots; ++s)
        if (h->owner[s] >= 0 && h->stamp[s] != step) cand.push_back(s);
    std::sort(cand.begin() + (std::ptrdiff_t)n_free, cand.end(), [&](int64_t x, int64_t y) {
        return h->stamp[x] != h->stamp[y] ? h->stamp[x] < h->stamp[y] : x < y;
    });
    int64_t taken = 0, ev = 0;
    size_t next = 0;
    for (int64_t e = 0; e < n && taken < max_plan; ++e) {
        if (touch[e] != step || h->table[e] >= 0) continue;
        if (grow_from && e % h->stride >= grow_from[e / h->stride]) continue;
        if (next >= cand.size()) break;  // every slot holds a page of this step
        const int64_t s = cand[next++];
        if (h->owner[s] >= 0) {
            h->table[h->owner[s]] = -1;
            ++ev;
        }
        h->owner[s] = e;
        h->stamp[s] = step;
        h->table[e] = (int32_t)s;
        plan[3 * taken] = (int32_t)(e / h->stride);
        plan[3 * taken + 1] = (int32_t)(e % h->stride);
        plan[3 * taken + 2] = (int32_t)s;
        ++taken;
    }
    if (n_in) *n_in = taken;
    if (n_evicted) *n_evicted = ev;
    return CSA_OK;
}

csa_status csa_hisparse_plan(csa_hisparse* h, const uint32_t* touch, uint32_t step, int32_t* plan, int64_t max_plan,
                             int64_t* n_in, int64_t* n_evicted) {
    if (!h || !touch || (max_plan > 0 && !plan) || max_plan < 0) return CSA_ERR_INVALID_ARG;
    return plan_impl(h, touch, step, plan, max_plan, n_in, n_evicted, nullptr);
}

csa_status csa_hisparse_update(csa_hisparse* h, const csa_decode_params* p, void* stream, int64_t* n_in,
                               int64_t* n_evicted) {
    if (!h || !p || !p->hs_ws_pool || !p->hs_ws_table || !p->hs_touch || !p->c_page_table || !p->kv_c)
        return CSA_ERR_INVALID_ARG;
    if (p->B != h->B || p->c_page_table_stride != h->stride || p->hs_n_slots != h->n_slots) return CSA_ERR_INVALID_ARG;
    int32_t* st = device_status_ptr();
    if (!st) return CSA_ERR_CUDA;
    if (h->swap_pending) {  // an asynchronous apply's uploads read the coordinator's buffers
        if (cudaEventSynchronize(h->ev_swap) != cudaSuccess) return CSA_ERR_CUDA;
        h->swap_pending = false;
    }
    if (!h->d_plan && cudaMalloc(&h->d_plan, (size_t)h->n_slots * 3 * sizeof(int32_t)) != cudaSuccess)
        return CSA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t n = (size_t)h->B * h->stride;
    if (cudaMemcpyAsync(h->touch.data(), p->hs_touch, n * sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return CSA_ERR_CUDA;
    h->plan.resize((size_t)h->n_slots * 3);
    int64_t taken = 0, ev = 0;
    csa_status rc = csa_hisparse_plan(h, h->touch.data(), p->hs_step, h->plan.data(), h->n_slots, &taken, &ev);
    if (rc) return rc;
    if (taken > 0) {
        if (cudaMemcpyAsync(h->d_plan, h->plan.data(), (size_t)taken * 3 * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return CSA_ERR_CUDA;
        hisparse_swap_kernel<<<(unsigned)taken, 256, 0, s>>>(h->d_plan, static_cast<const uint8_t*>(p->kv_c),
                                                            p->c_page_table, p->c_page_table_stride, p->c_n_pages,
                                                            p->c_page_stride, static_cast<uint8_t*>(p->hs_ws_pool), st);
        if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
        if (cudaMemcpyAsync(p->hs_ws_table, h->table.data(), n * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
            return CSA_ERR_CUDA;
    }
    if (n_in) *n_in = taken;
    if (n_evicted) *n_evicted = ev;
    return CSA_OK;
}

// The pinned buffers and events of the asynchronous form, made on first use.
static csa_status async_setup(csa_hisparse* h) {
    if (h->h_touch) return CSA_OK;
    const size_t n = (size_t)h->B * h->stride;
    if (!h->d_plan && cudaMalloc(&h->d_plan, (size_t)h->n_slots * 3 * sizeof(int32_t)) != cudaSuccess)
        return CSA_ERR_CUDA;
    if (cudaHostAlloc(&h->h_touch, n * sizeof(uint32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&h->h_table_evict, n * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&h->h_table_install, n * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc(&h->h_plan, (size_t)h->n_slots * 3 * sizeof(int32_t), cudaHostAllocDefault) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_touch, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_evict, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h->ev_swap, cudaEventDisableTiming) != cudaSuccess)
        return CSA_ERR_CUDA;
    return CSA_OK;
}

static csa_status check_update_args(const csa_hisparse* h, const csa_decode_params* p) {
    if (!h || !p || !p->hs_ws_pool || !p->hs_ws_table || !p->hs_touch || !p->c_page_table || !p->kv_c)
        return CSA_ERR_INVALID_ARG;
    if (p->B != h->B || p->c_page_table_stride != h->stride || p->hs_n_slots != h->n_slots) return CSA_ERR_INVALID_ARG;
    return CSA_OK;
}

csa_status csa_hisparse_collect(csa_hisparse* h, const csa_decode_params* p, void* stream) {
    csa_status rc = check_update_args(h, p);
    if (rc) return rc;
    if ((rc = async_setup(h))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t n = (size_t)h->B * h->stride;
    // a collect after an unapplied one replaces it: its event is recorded again below
    if (cudaMemcpyAsync(h->h_touch, p->hs_touch, n * sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaEventRecord(h->ev_touch, s) != cudaSuccess)
        return CSA_ERR_CUDA;
    h->collected_step = p->hs_step;
    h->collected = true;
    return CSA_OK;
}

csa_status csa_hisparse_apply(csa_hisparse* h, const csa_decode_params* p, const int64_t* n_tokens_host,
                              void* stream, void* side_stream, int64_t* n_in, int64_t* n_evicted) {
    csa_status rc = check_update_args(h, p);
    if (rc) return rc;
    if (!h->collected || !n_tokens_host || p->ratio < 1 || p->c_rows_per_page < 1) return CSA_ERR_INVALID_ARG;
    int32_t* st = device_status_ptr();
    if (!st) return CSA_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream), side = static_cast<cudaStream_t>(side_stream);
    const size_t n = (size_t)h->B * h->stride;
    // the stamps (usually landed long ago) and the previous apply's uploads, which read the
    // pinned buffers rewritten below
    if (cudaEventSynchronize(h->ev_touch) != cudaSuccess) return CSA_ERR_CUDA;
    if (h->swap_pending && cudaEventSynchronize(h->ev_swap) != cudaSuccess) return CSA_ERR_CUDA;
    h->swap_pending = false;
    h->collected = false;
    h->plan.resize((size_t)h->n_slots * 3);
    // the page holding each request's newest compressed row (and any later one) can still be
    // written by the steps this swap overlaps: it stays in the mirror
    std::vector<int64_t> grow((size_t)h->B);
    for (int32_t b = 0; b < h->B; ++b) {
        const int64_t G = n_tokens_host[b] / p->ratio;
        grow[(size_t)b] = G > 0 ? (G - 1) / p->c_rows_per_page : 0;
    }
    int64_t taken = 0, ev = 0;
    rc = plan_impl(h, h->h_touch, h->collected_step, h->plan.data(), h->n_slots, &taken, &ev, grow.data());
    if (rc) return rc;
    if (n_in) *n_in = taken;
    if (n_evicted) *n_evicted = ev;
    if (taken == 0) return CSA_OK;
    // 1. evictions first, on the decode stream: steps enqueued after this read those pages from
    //    the mirror, so no step reads a slot while it is refilled
    std::memcpy(h->h_table_install, h->table.data(), n * sizeof(int32_t));
    std::memcpy(h->h_table_evict, h->table.data(), n * sizeof(int32_t));
    for (int64_t i = 0; i < taken; ++i)  // the incoming pages stay in the mirror until installed
        h->h_table_evict[(int64_t)h->plan[3 * i] * h->stride + h->plan[3 * i + 1]] = -1;
    std::memcpy(h->h_plan, h->plan.data(), (size_t)taken * 3 * sizeof(int32_t));
    if (cudaMemcpyAsync(p->hs_ws_table, h->h_table_evict, n * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaEventRecord(h->ev_evict, s) != cudaSuccess)
        return CSA_ERR_CUDA;
    // 2. on the side stream, overlapping the next steps: the pages into their slots, then the
    //    installed table (an entry only ever goes from -1 to a slot whose bytes are in place)
    if (cudaStreamWaitEvent(side, h->ev_evict, 0) != cudaSuccess ||
        cudaMemcpyAsync(h->d_plan, h->h_plan, (size_t)taken * 3 * sizeof(int32_t), cudaMemcpyHostToDevice, side) !=
            cudaSuccess)
        return CSA_ERR_CUDA;
    hisparse_swap_kernel<<<(unsigned)taken, 256, 0, side>>>(h->d_plan, static_cast<const uint8_t*>(p->kv_c),
                                                            p->c_page_table, p->c_page_table_stride, p->c_n_pages,
                                                            p->c_page_stride, static_cast<uint8_t*>(p->hs_ws_pool), st);
    if (cudaGetLastError() != cudaSuccess) return CSA_ERR_CUDA;
    if (cudaMemcpyAsync(p->hs_ws_table, h->h_table_install, n * sizeof(int32_t), cudaMemcpyHostToDevice, side) !=
            cudaSuccess ||
        cudaEventRecord(h->ev_swap, side) != cudaSuccess)
        return CSA_ERR_CUDA;
    h->swap_pending = true;
    return CSA_OK;
}

}  // extern "C"
