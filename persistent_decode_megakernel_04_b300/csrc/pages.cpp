// pages.cpp — host-side allocator of the paged KV cache for continuous
// batching (declared in include/mk.h).
//
// A plan's batch is a fixed set of rows; between decode steps sequences are
// admitted into free rows, grow page by page, and retire, their pages going
// back to the pool for the next sequence.  This is the serving regime of the
// high-throughput megakernel ("Llama-70B 向け…megakernel", section
// 高スループットMegakernelの設計と工夫: large batches of sequences of
// different lengths), kept on one GPU.
//
// The last page of the pool is reserved as scratch: every entry of a free
// row points at it, so that a decode step over the whole batch can run a
// free row (token 0 at position 0) without touching any sequence's pages.
#include <cuda_runtime.h>

#include <cstring>
#include <new>
#include <vector>

#include "../../include/mk.h"

struct mk_page_pool {
    int32_t num_pages = 0, batch = 0, max_pages = 0, page_size = 0;
    int32_t scratch = 0;              // page every free row's entries point at
    std::vector<int32_t> free_pages;  // stack of free page ids
    std::vector<int32_t> table;       // [batch][max_pages], host copy of the page table
    std::vector<int32_t> held;        // pages held by each row (its first held[row] entries)
    std::vector<uint8_t> live;        // row admitted
    bool dirty = true;                // host table changed since the last sync
};

namespace {

mk_status grow(mk_page_pool *p, int32_t row, int32_t n_tokens) {
    const int32_t need = (n_tokens + p->page_size - 1) / p->page_size;
    if (need > p->max_pages) return MK_ERR_INVALID;
    if (need - p->held[row] > (int32_t)p->free_pages.size()) return MK_ERR_OOM;
    for (int32_t j = p->held[row]; j < need; ++j) {
        p->table[(size_t)row * p->max_pages + j] = p->free_pages.back();
        p->free_pages.pop_back();
        p->dirty = true;
    }
    if (need > p->held[row]) p->held[row] = need;
    return MK_OK;
}

}  // namespace

extern "C" {

mk_status mk_pages_create(int32_t num_pages, int32_t batch, int32_t max_pages_per_seq, int32_t page_size,
                          mk_page_pool **out) {
    if (!out || num_pages < 2 || batch <= 0 || max_pages_per_seq <= 0 || page_size <= 0) return MK_ERR_INVALID;
    *out = nullptr;
    mk_page_pool *p = new (std::nothrow) mk_page_pool();
    if (!p) return MK_ERR_OOM;
    p->num_pages = num_pages;
    p->batch = batch;
    p->max_pages = max_pages_per_seq;
    p->page_size = page_size;
    p->scratch = num_pages - 1;
    // lowest ids handed out first
    for (int32_t i = num_pages - 2; i >= 0; --i) p->free_pages.push_back(i);
    p->table.assign((size_t)batch * max_pages_per_seq, p->scratch);
    p->held.assign(batch, 0);
    p->live.assign(batch, 0);
    *out = p;
    return MK_OK;
}

mk_status mk_pages_admit(mk_page_pool *p, int32_t row, int32_t n_tokens) {
    if (!p || row < 0 || row >= p->batch || n_tokens <= 0 || p->live[row]) return MK_ERR_INVALID;
    const mk_status st = grow(p, row, n_tokens);
    if (st != MK_OK) return st;
    p->live[row] = 1;
    return MK_OK;
}

mk_status mk_pages_extend(mk_page_pool *p, int32_t row, int32_t n_tokens) {
    if (!p || row < 0 || row >= p->batch || !p->live[row] || n_tokens <= 0) return MK_ERR_INVALID;
    return grow(p, row, n_tokens);
}

mk_status mk_pages_retire(mk_page_pool *p, int32_t row) {
    if (!p || row < 0 || row >= p->batch || !p->live[row]) return MK_ERR_INVALID;
    for (int32_t j = p->held[row] - 1; j >= 0; --j) {
        int32_t &e = p->table[(size_t)row * p->max_pages + j];
        p->free_pages.push_back(e);
        e = p->scratch;
    }
    p->held[row] = 0;
    p->live[row] = 0;
    p->dirty = true;
    return MK_OK;
}

int32_t mk_pages_free_count(const mk_page_pool *p) { return p ? (int32_t)p->free_pages.size() : -1; }

int32_t mk_pages_scratch_page(const mk_page_pool *p) { return p ? p->scratch : -1; }

mk_status mk_pages_table(const mk_page_pool *p, int32_t *out, int64_t capacity) {
    if (!p || !out || capacity < (int64_t)p->table.size()) return MK_ERR_INVALID;
    std::memcpy(out, p->table.data(), p->table.size() * sizeof(int32_t));
    return MK_OK;
}

mk_status mk_pages_sync(mk_page_pool *p, int32_t *page_table_dev, void *stream) {
    if (!p || !page_table_dev) return MK_ERR_INVALID;
    if (!p->dirty) return MK_OK;
    // pageable source: the call returns once the table has been staged, so
    // the host copy may change again right away
    const cudaError_t e = cudaMemcpyAsync(page_table_dev, p->table.data(), p->table.size() * sizeof(int32_t),
                                          cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MK_ERR_CUDA;
    }
    p->dirty = false;
    return MK_OK;
}

void mk_pages_destroy(mk_page_pool *p) { delete p; }

}  // extern "C"
