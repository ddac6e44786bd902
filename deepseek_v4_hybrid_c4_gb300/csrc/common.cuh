// Device-side helpers shared by the libcsa kernels: paged-row addressing, the
// sticky status word, the order-preserving score key, bf16 packing.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "csa.h"
#include "ptx.cuh"

namespace csa {

constexpr int D = 512;        // latent dim (K = V row), bf16 -> 1024 B per row
constexpr int DI = 128;       // index-key dim
constexpr int ROW_BYTES = D * 2;

// A paged row buffer as the kernels see it (see csa_paged in csa.h).  For a
// batch, request b uses page_table + (b / qpr) * pt_stride: with speculative verify a
// batch entry is one query position and qpr positions share their request's table.
struct DPaged {
    const uint8_t* base;
    const int32_t* pt;   // nullptr -> contiguous (physical page = logical page)
    int64_t pt_stride;   // int32 entries between requests' page tables
    int64_t page_stride; // bytes
    int64_t n_pages;
    int32_t rpp;         // rows per page
    int32_t qpr;         // batch entries per page table (>= 1)
};

// HiSparse working set over a paged pool whose rows live in a host mirror: table[(b / qpr) *
// pt_stride + logical page] is the GPU slot holding that page (slots of the pool's page stride at
// base), or -1 -- the row is then read from the pool itself, host memory mapped into the device's
// address space.  touch, when set, gets `step` for every page read (the LRU stamps).
struct DWorkSet {
    const int32_t* table;  // nullptr: no working set
    uint8_t* base;
    int64_t n_slots;
    uint32_t* touch;
    uint32_t step;
};

// Tokens visible to batch entry q of a decode step whose requests carry nq query positions
// each (speculative verify: the draft tokens are the last nq of request q / nq, and query j
// sits at position n_tokens - nq + j, so it sees n_tokens - nq + j + 1 tokens).
CSA_DEV int64_t query_tokens(const int64_t* n_tokens, int q, int nq) {
    if (nq <= 1) return __ldg(n_tokens + q);
    const int b = q / nq;
    return __ldg(n_tokens + b) - nq + (q - b * nq) + 1;
}

// Record an error code in the sticky device status word (bit code-1).
CSA_DEV void raise_status(int32_t* status, int code) {
    if (status) atomicOr(status, 1 << (code - 1));
}

// Address of logical row r of request b, or nullptr (and CSA_ERR_DEVICE_BOUNDS) when
// its page id falls outside the pool.
CSA_DEV const uint8_t* row_addr(const DPaged& p, int b, int64_t r, int row_bytes, int32_t* status) {
    const int64_t lp = r / p.rpp;
    const int64_t slot = r - lp * p.rpp;
    int64_t pp = lp;
    if (p.pt) pp = __ldg(p.pt + (int64_t)(p.qpr > 1 ? b / p.qpr : b) * p.pt_stride + lp);
    if (pp < 0 || pp >= p.n_pages) {
        raise_status(status, CSA_ERR_DEVICE_BOUNDS);
        return nullptr;
    }
    return p.base + pp * p.page_stride + slot * (int64_t)row_bytes;
}

// Row r of request b in its working-set slot, or nullptr when the page is not resident.
CSA_DEV uint8_t* ws_slot_row(const DWorkSet& w, const DPaged& p, int b, int64_t r) {
    if (!w.table) return nullptr;
    const int64_t lp = r / p.rpp;
    const int32_t sl = w.table[(int64_t)(p.qpr > 1 ? b / p.qpr : b) * p.pt_stride + lp];
    return sl >= 0 && sl < w.n_slots ? w.base + sl * p.page_stride + (r - lp * p.rpp) * (int64_t)ROW_BYTES : nullptr;
}

// Row r of request b of a pool with a working set: its GPU slot when resident, else the pool's
// own row; stamps the page when `stamp` and the set keeps stamps.
CSA_DEV const uint8_t* ws_row(const DWorkSet& w, const DPaged& p, int b, int64_t r, bool stamp, int32_t* status) {
    if (w.table) {
        const int64_t lp = r / p.rpp;
        const int64_t e = (int64_t)(p.qpr > 1 ? b / p.qpr : b) * p.pt_stride + lp;
        if (stamp && w.touch) w.touch[e] = w.step;
        const int32_t sl = w.table[e];
        if (sl >= 0 && sl < w.n_slots) return w.base + sl * p.page_stride + (r - lp * p.rpp) * (int64_t)ROW_BYTES;
    }
    return row_addr(p, b, r, ROW_BYTES, status);
}

// Order-preserving 32-bit image of an fp32 score: larger score <-> larger key,
// -0 and +0 map to the same key.
CSA_DEV uint32_t score_key(float s) {
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

CSA_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
CSA_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

CSA_DEV uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace csa
